"""A CPU model of the column-group kernels' arithmetic (k_planes_cg and
k_planes_cg_reduce): their tiles of whole rows, items of several planes over
several tiles, tiles that start inside a 16-byte granule, idle threads past the
row groups, per-thread runs with one plane boundary at most, segmented scans
over the lanes of one column group, per-(warp, group) head flags and the carry
from tile to tile -- written out in Python with the kernels' index formulas and
run on small integer inputs, where every result is exact, against the oracle.
It guards the scheme the kernels implement; the kernels themselves are checked
on the GPU against the same oracle."""
import numpy as np
import pytest

import oracle

T, NW = 128, 4  # threads and warps per block


def shape_of(P):
    """Group width V, run rows S, groups G, row groups RG and tile rows TR."""
    V = 4 if P % 4 == 0 else 2 if P % 2 == 0 else 1
    S = {4: 9, 2: 17, 1: 33}[V]
    G = P // V
    RG = T // G
    return V, S, G, RG, RG * S


def plan(outer, N, P, per):
    """Planes per item (items of up to `per` tiles) and ceil(2^32 / N)."""
    _, _, _, _, TR = shape_of(P)
    k = TR * per // N
    k = k if k >= 2 else 1
    return k, ((1 << 32) + N - 1) // N


def head(rr, N, S, k, magic, rev):
    """Scan position of the first plane boundary in a run of S rows starting
    at item-relative row rr (S when none), and for a forward walk the plane
    that ends in the run: (dd, q) with its last row dd - 1 rows in."""
    hp, dd, q = S, 0, 0
    if k == 1:
        if not rev:
            d = 0 if rr == 0 else N - rr
            hp = d if 0 <= d < S else S
            if rr > 0 and 1 <= d <= S:
                dd, q = d, 1
        else:
            e = rr + S - N
            hp = e if 0 <= e < S else S
    else:
        if not rev:
            q = 0 if rr == 0 else (((rr - 1) * magic) >> 32) + 1
            assert q == -(-rr // N)
            d = q * N - rr
            hp = d if d < S else S
            if q >= 1 and 1 <= d <= S:
                dd = d
            else:
                q = 0
        else:
            gq = rr + S
            qq = (gq * magic) >> 32
            assert qq == gq // N
            e = gq - qq * N
            hp = e if qq >= 1 and e < S else S
    return hp, dd, q


def lane_fold(values, heads, w, G):
    """Segmented inclusive scan over each column group's lanes of warp w:
    inclusive values, the value of the group's previous lane, whether a head
    lies before, and the group's last-lane total and head flag."""
    inc, prev, before, last = {}, {}, {}, {}
    for g in range(G):
        lanes = [l for l in range(32) if (32 * w + l) % G == g]
        run, any_head = None, False
        for i, l in enumerate(lanes):
            t = 32 * w + l
            prev[t] = run
            before[t] = any_head
            run = values[t] if (run is None or heads[t]) else (run + values[t]).astype(np.float32)
            any_head = any_head or heads[t]
            inc[t] = run
        last[g] = (run, any_head)
    return inc, prev, before, last


def model(x, outer, N, P, rev=False, excl=False, reduce=False, per=1, grid=3):
    V, S, G, RG, TR = shape_of(P)
    assert N > S and not (reduce and rev)
    L = N * P
    k, magic = plan(outer, N, P, per)
    items = -(-outer // k)
    n = outer * L
    xpad = np.zeros(((n + 3) // 4) * 4, np.float32)
    xpad[:n] = x
    y = np.full(outer * P if reduce else n, np.nan, np.float32)
    written = np.zeros(y.shape, np.int64)
    for b in range(grid):
        buf = np.full(T * S * V + 8, np.nan, np.float32)  # stale contents are NaN
        for item in range(b, items, grid):
            first = item * k
            planes = min(k, outer - first)
            lo, rows_item = first * L, planes * N
            tiles = -(-rows_item // TR)
            carry = np.zeros((G, V), np.float32)
            for j in range(tiles):
                jt = tiles - 1 - j if rev else j
                tr0 = jt * TR
                rows = min(TR, rows_item - tr0)
                f0 = lo + tr0 * P
                a0, a1 = f0 & ~3, (f0 + rows * P + 3) & ~3
                delta = f0 - a0
                buf[: a1 - a0] = xpad[a0:a1]
                acc = np.zeros((T, V), np.float32)
                pre = np.zeros((T, V), np.float32)
                vals = np.zeros((T, S, V), np.float32)
                hps, ends = np.full(T, S), {}
                for t in range(RG * G):
                    g = t % G
                    m = RG - 1 - t // G if rev else t // G
                    hp, dd, q = head(tr0 + m * S, N, S, k, magic, rev)
                    hps[t] = hp
                    if dd:
                        ends[t] = q
                    a = np.zeros(V, np.float32)
                    for e in range(S):
                        row = m * S + (S - 1 - e if rev else e)
                        v = buf[delta + row * P + V * g: delta + row * P + V * g + V]
                        before = np.zeros(V, np.float32) if e == hp else a
                        a = (before + v).astype(np.float32)
                        vals[t, e] = before if excl else a
                        if e < hp:
                            pre[t] = a
                    acc[t] = a
                # lane scans per warp and group, then the warps in order
                new_carry = np.zeros_like(carry)
                warp_tot = {}
                for w in range(NW):
                    inc, prev, bef, last = lane_fold(acc, {t: hps[t] < S for t in range(T)}, w, G)
                    warp_tot[w] = (inc, prev, bef, last)
                for t in range(T):
                    w, l, g = t // 32, t % 32, t % G
                    cw = carry[g].copy()
                    for q in range(w):
                        tot, flag = warp_tot[q][3][g]
                        cw = tot.copy() if flag else (cw + tot).astype(np.float32)
                    if w == NW - 1 and l >= 32 - G:
                        tot, flag = warp_tot[w][3][g]
                        new_carry[g] = tot if flag else (cw + tot).astype(np.float32)
                    if t >= RG * G:
                        continue
                    _, prev, bef, _ = warp_tot[w]
                    cl = cw if l < G else (prev[t] if bef[t] else (cw + prev[t]).astype(np.float32))
                    m = RG - 1 - t // G if rev else t // G
                    if reduce:
                        if t in ends and ends[t] <= planes:
                            out = (first + ends[t] - 1) * P + V * g
                            y[out: out + V] = (cl + pre[t]).astype(np.float32)
                            written[out: out + V] += 1
                        continue
                    for e in range(S):
                        row = m * S + (S - 1 - e if rev else e)
                        o = delta + row * P + V * g
                        buf[o: o + V] = (cl + vals[t, e]).astype(np.float32) if e < hps[t] else vals[t, e]
                carry = new_carry
                if not reduce:
                    y[f0: f0 + rows * P] = buf[delta: delta + rows * P]
                    written[f0: f0 + rows * P] += 1
    assert (written == 1).all(), "every output written exactly once"
    return y


# Single floats, float2 and float4 groups; planes of one run and a row; one
# plane over several tiles; 128 columns (32 groups); items of many planes
# over 2-3 tiles (the last three).
CASES = [(3, 40, 11, 1), (5, 18, 18, 1), (4, 100, 20, 1), (2, 300, 13, 1), (1, 700, 16, 1),
         (3, 50, 128, 1), (40, 34, 11, 3), (70, 10, 12, 2), (250, 20, 6, 3)]


@pytest.mark.parametrize("outer,N,P,per", CASES)
@pytest.mark.parametrize("rev,excl", [(False, False), (True, False), (False, True), (True, True)])
def test_scan_model_matches_oracle(outer, N, P, per, rev, excl):
    x = np.random.default_rng(outer * 1000 + N + P).integers(-3, 4, size=outer * N * P).astype(np.float32)
    got = model(x, outer, N, P, rev=rev, excl=excl, per=per)
    ref, _ = oracle.cumsum(x, outer, N, P, rev, excl)
    assert np.array_equal(got, np.asarray(ref).reshape(-1))


@pytest.mark.parametrize("outer,N,P,per", CASES)
def test_reduce_model_matches_oracle(outer, N, P, per):
    x = np.random.default_rng(outer * 1000 + N + P + 1).integers(-3, 4, size=outer * N * P).astype(np.float32)
    got = model(x, outer, N, P, reduce=True, per=per)
    ref, _ = oracle.axis_sum(x, outer, N, P)
    assert np.array_equal(got, np.asarray(ref).reshape(-1))
