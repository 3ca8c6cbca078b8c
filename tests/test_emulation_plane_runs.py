"""A CPU model of the plane-run kernel's arithmetic (k_planes, 2 to 14
columns): tiles from the item's start rounded down to lcm(4, P) floats, runs
of whole rows per thread with the column class of every float known, heads
from one multiply-shift division (planes many to a tile), the position walk of
planes no longer than a run (several boundaries in a run), the warp fast path,
segmented lane scans per class, the warp fold and the carry from tile to tile,
reductions writing each plane's totals where it ends -- written out in Python
with the kernel's index formulas and run on small integer inputs, where every
result is exact, against the oracle.  Stale shared memory is NaN, so a read of
it shows.  The kernel itself is checked on the GPU against the same oracle."""
import numpy as np
import pytest

import oracle

T = 128
NW = 4


def runlen(P):
    return {5: 20, 7: 28, 8: 24, 10: 20, 14: 28}.get(P, 36)


def align(P):
    return {3: 12, 6: 12, 12: 12, 5: 20, 7: 28, 8: 8, 9: 36, 10: 20, 14: 28}.get(P, 4)


def plan(outer, N, P):
    L = N * P
    R = runlen(P)
    TL = T * R
    assert N >= 2
    k = (TL - align(P) + 1) // L
    k = k if k >= 2 else 1
    items = -(-outer // k)
    magic = ((1 << 32) + L - 1) // L if k >= 2 else 0
    return k, items, magic


def item_of(i, k, outer, L, P):
    TL = T * runlen(P)
    first = i * k
    planes = min(k, outer - first)
    lo = first * L
    hi = lo + planes * L
    vlo = lo - lo % align(P)
    tiles = -(-(hi - vlo) // TL)
    return lo, hi, vlo, first, planes, tiles


def rel_sat(a, b):
    far = 1 << 30
    return max(min(a - b, far), -far)


def run(x, outer, N, P, scan=True, rev=False, excl=False, grid=7):
    R = runlen(P)
    TL = T * R
    n = outer * N * P
    L = N * P
    k, items, magic = plan(outer, N, P)
    xf = np.asarray(x, dtype=np.float32).reshape(-1)
    # allocation padded to a granule with garbage
    xpad = np.full(((n + 3) // 4) * 4, np.float32(np.nan), dtype=np.float32)
    xpad[:n] = xf
    y = np.full(n if scan else outer * P, np.nan, dtype=np.float32)
    written = np.zeros(y.shape, dtype=np.int64)
    for b in range(grid):
        bufs = [np.full(TL, np.nan, dtype=np.float32) for _ in range(3)]
        stage = 0
        carry_prev = None
        item = b
        while item < items:
            lo, hi, vlo, first, planes, tiles = item_of(item, k, outer, L, P)
            for j in range(tiles):
                mt = tiles - 1 - j if rev else j
                ts = vlo + mt * TL
                te = min(ts + TL, (hi + 3) & ~3)
                assert te > ts and (te - ts) % 4 == 0 and ts % 4 == 0 and ts >= 0
                assert te <= len(xpad)
                buf = bufs[stage]
                buf[: te - ts] = xpad[ts:te]   # the rest stays as the previous tile left it
                rlo = rel_sat(lo, ts)
                rhi = rel_sat(hi, ts)
                # per thread
                v = np.zeros((T, R), dtype=np.float32)
                hp = np.full(T, R, dtype=np.int64)
                dd = np.full(T, -1, dtype=np.int64)
                qf = np.zeros(T, dtype=np.int64)
                avec = np.zeros(T, dtype=np.int64)
                pos0 = np.zeros(T, dtype=np.int64)
                qfirst = np.zeros(T, dtype=np.int64)
                hlast = np.zeros(T, dtype=np.int64)
                ends = [[] for _ in range(T)]
                for t in range(T):
                    a = (T - 1 - t if rev else t) * R
                    avec[t] = a
                    mem = buf[a:a + R]
                    v[t] = mem[::-1] if rev else mem
                    if L <= R:
                        rr = a - rlo
                        u = rr + (R - 1 if rev else 0) + 64 * L
                        assert 0 < u < (1 << 32) // L
                        q = (u * magic) >> 32
                        assert q == u // L
                        pos0[t] = u - q * L
                        qfirst[t] = q - 64
                        hf = (0 if pos0[t] + 1 == L else pos0[t] + 1) if rev else (0 if pos0[t] == 0 else L - pos0[t])
                        hp[t] = hf
                        hlast[t] = hf + L * ((((R - 1 - hf) * magic) >> 32))
                        assert hlast[t] == hf + L * ((R - 1 - hf) // L)
                    elif k == 1:
                        if not rev:
                            d1, d2 = rlo - a, rhi - a
                            if 0 <= d1 < R:
                                hp[t] = d1
                            elif 0 <= d2 < R:
                                hp[t] = d2
                            if 1 <= d2 <= R:
                                dd[t] = d2
                                qf[t] = 1
                        else:
                            e = a + R - rhi
                            if 0 <= e < R:
                                hp[t] = e
                    else:
                        assert 0 <= rlo < align(P)
                        rr = a - rlo
                        if not rev:
                            q = 0 if rr <= 0 else (((rr - 1) * magic) >> 32) + 1
                            assert q == (0 if rr <= 0 else -(-rr // L))
                            d = q * L - rr
                            assert d >= 0
                            if d < R:
                                hp[t] = d
                            if 1 <= d <= R:
                                dd[t] = d
                            qf[t] = q
                        else:
                            g = rr + R
                            qr = (g * magic) >> 32
                            assert qr == g // L
                            e = g - qr * L
                            if qr >= 1 and e < R:
                                hp[t] = e
                # 1. local scan (as the kernel: per-warp fast path, else restart rule)
                acc = np.zeros((T, P), dtype=np.float32)
                pre = np.zeros((T, P), dtype=np.float32)
                outv = v.copy()
                for w in range(NW):
                    if L <= R:
                        for t in range(w * 32, w * 32 + 32):
                            pos = pos0[t]
                            for e in range(R):
                                c = e % P
                                restart = (pos >= L - P) if rev else (pos < P)
                                before = np.float32(0) if restart else acc[t, c]
                                acc[t, c] = v[t, e] if restart else np.float32(acc[t, c] + v[t, e])
                                if scan:
                                    outv[t, e] = before if excl else acc[t, c]
                                else:
                                    outv[t, e] = acc[t, c]
                                    if pos == L - 1:
                                        ends[t].append(e)
                                pos = (L - 1 if pos == 0 else pos - 1) if rev else (0 if pos + 1 == L else pos + 1)
                            hl = hlast[t]
                            for c in range(P):
                                if hl + ((c - hl % P + P) % P) >= R:
                                    acc[t, c] = 0
                        continue
                    fast = not any(0 < hp[t] < R for t in range(w * 32, w * 32 + 32))
                    for t in range(w * 32, w * 32 + 32):
                        for e in range(R):
                            c = e % P
                            if fast:
                                before = acc[t, c]
                                acc[t, c] = np.float32(acc[t, c] + v[t, e])
                            else:
                                restart = 0 <= e - hp[t] < P
                                before = np.float32(0) if restart else acc[t, c]
                                acc[t, c] = v[t, e] if restart else np.float32(acc[t, c] + v[t, e])
                                if e < hp[t]:
                                    pre[t, c] = acc[t, c]
                            outv[t, e] = before if excl else acc[t, c]
                        if fast:
                            if hp[t] == R:
                                pre[t] = acc[t]
                        else:
                            for c in range(P):
                                if R - P + c < hp[t] < R:
                                    acc[t, c] = 0
                # 2. lane scan per warp
                inc = acc.copy()
                ex = np.zeros_like(acc)
                head_before = np.zeros(T, dtype=bool)
                wagg = np.zeros((NW, P), dtype=np.float32)
                wflag = np.zeros(NW, dtype=bool)
                for w in range(NW):
                    lanes = range(w * 32, w * 32 + 32)
                    hmask = [hp[t] < R for t in lanes]
                    hh = []
                    for l in range(32):
                        hs = [i for i in range(l + 1) if hmask[i]]
                        hh.append(hs[-1] if hs else 0)
                    cur = inc[w * 32:(w + 1) * 32].copy()
                    o = 1
                    while o < 32:
                        nxt = cur.copy()
                        for l in range(32):
                            src = l - o
                            if src >= hh[l]:
                                nxt[l] = (cur[src] + cur[l]).astype(np.float32)
                        cur = nxt
                        o <<= 1
                    inc[w * 32:(w + 1) * 32] = cur
                    for l in range(32):
                        t = w * 32 + l
                        ex[t] = cur[l - 1] if l > 0 else cur[l]
                        head_before[t] = any(hmask[:l])
                    wagg[w] = cur[31]
                    wflag[w] = any(hmask)
                # 3. warp carries
                cw_all = np.zeros((NW, P), dtype=np.float32)
                c0 = np.zeros(P, dtype=np.float32) if j == 0 else carry_prev
                cw = c0.copy()
                for w in range(NW):
                    cw_all[w] = cw
                    cw = wagg[w].copy() if wflag[w] else (cw + wagg[w]).astype(np.float32)
                carry_prev = cw
                for t in range(T):
                    w, l = t // 32, t % 32
                    if l == 0:
                        cl = cw_all[w]
                    elif head_before[t]:
                        cl = ex[t]
                    else:
                        cl = (cw_all[w] + ex[t]).astype(np.float32)
                    if scan:
                        for e in range(R):
                            if e < hp[t]:
                                outv[t, e] = np.float32(cl[e % P] + outv[t, e])
                        a = avec[t]
                        buf[a:a + R] = outv[t][::-1] if rev else outv[t]
                    elif L <= R:
                        q = qfirst[t]
                        for e in ends[t]:
                            if 0 <= q < planes:
                                plane = first + q
                                for c in range(P):
                                    idx = e - ((e % P - c + P) % P)
                                    if idx < 0:
                                        val = cl[c]
                                    elif idx < hp[t]:
                                        val = np.float32(cl[c] + outv[t, idx])
                                    else:
                                        val = outv[t, idx]
                                    y[plane * P + c] = val
                                    written[plane * P + c] += 1
                            q += 1
                    else:
                        if dd[t] >= 1 and 1 <= qf[t] <= planes:
                            plane = first + qf[t] - 1
                            for c in range(P):
                                y[plane * P + c] = np.float32(cl[c] + pre[t, c])
                                written[plane * P + c] += 1
                if scan:
                    lo_t = min(max(rlo, 0), TL)
                    hi_t = min(max(rhi, 0), TL)
                    ga = (lo_t + 3) & ~3
                    gb = hi_t & ~3
                    if ga < gb:
                        for f in range(ga, gb):
                            y[ts + f] = buf[f]
                            written[ts + f] += 1
                    for tt in range(8):
                        f = lo_t + tt if tt < 4 else max(gb, ga) + (tt - 4)
                        lim = min(ga, hi_t) if tt < 4 else hi_t
                        if f < lim:
                            y[ts + f] = buf[f]
                            written[ts + f] += 1
                stage = (stage + 1) % 3
            item += grid
    assert (written == 1).all(), ("write count", np.unique(written, return_counts=True))
    return y


CASES = [(3, 100, 3), (17, 13, 2), (5, 767, 3), (40, 7, 3), (7, 4, 5), (3, 37, 10), (9, 101, 14),
         (25, 2, 12), (2, 2305, 2), (11, 9, 4), (6, 3, 8), (4, 1025, 9)]


@pytest.mark.parametrize("outer,N,P", CASES)
@pytest.mark.parametrize("rev,excl", [(False, False), (True, False), (False, True), (True, True)])
def test_scan_model_matches_oracle(outer, N, P, rev, excl):
    x = np.random.default_rng(outer * 1000 + N + P).integers(-3, 4, size=outer * N * P).astype(np.float32)
    got = run(x, outer, N, P, True, rev, excl)
    ref, _ = oracle.cumsum(x, outer, N, P, rev, excl)
    assert np.array_equal(got, np.asarray(ref).reshape(-1))


@pytest.mark.parametrize("outer,N,P", [c for c in CASES if c[2] <= 8])
def test_reduce_model_matches_oracle(outer, N, P):
    x = np.random.default_rng(outer * 1000 + N + P + 1).integers(-3, 4, size=outer * N * P).astype(np.float32)
    got = run(x, outer, N, P, False, False, False)
    ref, _ = oracle.axis_sum(x, outer, N, P)
    assert np.array_equal(got, np.asarray(ref).reshape(-1))
