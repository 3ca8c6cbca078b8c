// lr_planes.cuh -- cumulative sums and reductions along the middle axis of
// [outer, N, P] for narrow planes (sm_103a): reductions of 2 .. 8 columns,
// scans of 2 .. 128 columns.
//
// The POPCORNBENCH trace l1_p91 discusses scanning a dimension other than the
// last; here that dimension has stride P.  Read flat, plane o is the L = N*P
// consecutive floats from o*L, and the float at flat index f lies in column
// f % P (L is a multiple of P).  Scanning every plane along N is then P
// interleaved scans of the flat array, one per column class, each restarting
// at every plane boundary: a segmented scan whose segments are the planes.
// The reduction is the same walk that keeps only each plane's totals.
//
// Work is cut into items of k whole planes (k >= 2 short planes in one tile,
// or one plane over one or more tiles).  A block takes items in turn and
// processes an item's tiles in scan order, with a per-class carry from tile
// to tile.  A tile lands in shared memory by one bulk copy (TMA engine),
// three tiles in flight per block; its start is the item's start rounded
// down to a 16-byte boundary and a multiple of P.
//
// Thread t of the 128 owns run m of R consecutive floats of the tile (m = t;
// m = 127 - t for a reverse scan, whose scan order runs down memory): R = 36
// for 2, 3, 4, 6, 9 and 12 columns, 20 for 5 and 10, 28 for 7 and 14, 24 for
// 8 (kRunOf).  R holds whole rows and every run starts at a multiple of P, so
// the column class of each of a thread's floats is known at compile time.
// When L > R a run holds at most one plane boundary (its "head": the scan
// position where a plane starts, in scan order); planes no longer than a run
// take the MULTI form, which walks each float's position in its plane and
// restarts a class on its plane's first row.  The steps:
//   1. a sequential per-class scan over the run, restarting at the head;
//   2. a segmented shuffle scan of the run totals across the warp (per class,
//      the lanes before a lane's last head excluded);
//   3. the warps' totals through shared memory, folded in warp order with the
//      carry of the previous tile (same segment rule);
//   4. each float before its run's (first) head gets its lane's carry; a
//      scan writes the run back in place and the tile leaves by one bulk
//      store of its whole 16-byte granules (the item's partial first and
//      last granules by plain stores); a reduction writes the P totals of
//      each plane that ends in the run.
// Scans of other column counts, up to 128 (k_planes_cg), give thread t one
// column group (a float4, float2 or float) of a run of 9, 17 or 33 rows
// instead, so that its classes are the group's components.
// Every output is a sum over its own terms in a fixed order (an exclusive
// output leaves its own term out of the running value), nothing is
// subtracted, and reruns are bit-identical.  Floats of the tile outside the
// item (before its start, after its end) are loaded but fall in other
// segments, so they never reach an output; only the item's own floats are
// stored.
//
// The kernels are templates here; lr_planes_scan.cu, lr_planes_reduce.cu and
// lr_planes_lb.cu instantiate and launch the scans, the reductions and the
// look-back form (three translation units, compiled in parallel).
#pragma once

#include <algorithm>

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

constexpr int kT = kPlanesThreads;
constexpr int kNW = kT / 32;
// Floats per thread run for P columns: whole rows, a multiple of 4 (float4
// chunks) and, where P allows, an odd number of chunks, so that the runs of
// 8 consecutive threads fall in distinct shared-memory banks (8 columns: 6
// chunks, two threads to a bank).  At most 36, so that three tiles of four
// blocks fit an SM.
template <int P>
constexpr int kRunOf = planes_run_len(P);
template <int P>
constexpr int kTileOf = kT * kRunOf<P>;
template <int P>
constexpr int kChunksOf = kRunOf<P> / 4;
constexpr int kStages = 3;
constexpr int kLbBlocks = 6;  // resident look-back blocks per SM: 6 x 37 KB of tiles, <= 85 registers
// Runs and tiles start on multiples of this many floats: 16 bytes and P.
template <int P>
constexpr int kPlaneAlign = planes_align(P);

struct PlaneItem {
  int64_t lo, hi;  // the item's floats [lo, hi): planes first .. first + planes - 1
  int64_t vlo;     // lo rounded down to kPlaneAlign
  int64_t first;
  int planes;
  int tiles;       // tiles covering [vlo, hi)
};

template <int P>
__device__ __forceinline__ PlaneItem plane_item(const PlaneRunParams& p, int64_t i) {
  const int64_t L = p.N * P;
  PlaneItem it;
  it.first = i * p.k;
  const int64_t planes = min(p.k, p.outer - it.first);
  it.planes = (int)planes;
  it.lo = it.first * L;
  it.hi = it.lo + planes * L;
  it.vlo = it.lo - it.lo % kPlaneAlign<P>;
  it.tiles = (int)((it.hi - it.vlo + kTileOf<P> - 1) / kTileOf<P>);
  return it;
}

// The producer's position: the next tile to copy in, in the block's order
// (items blockIdx.x, blockIdx.x + gridDim.x, ...; each item's tiles in scan
// order).  Only thread 0 issues copies; the cursor lives in shared memory.
struct Cursor {
  int64_t item;
  int tile;
  PlaneItem it;
};

// The first float of scan-order tile j of an item.
template <int P>
__device__ __forceinline__ int64_t tile_start(const PlaneItem& it, int j, bool rev) {
  return it.vlo + (int64_t)(rev ? it.tiles - 1 - j : j) * kTileOf<P>;
}

template <int P>
__device__ __forceinline__ void issue_tile(const PlaneRunParams& p, Cursor& c, bool rev, float* buf,
                                           unsigned long long* bar) {
  if (c.item >= p.items) return;
  const int64_t ts = tile_start<P>(c.it, c.tile, rev);
  // Whole 16-byte granules up to the item's end: the last one lies in the
  // same page as the item's last float.
  const int64_t te = min(ts + kTileOf<P>, (c.it.hi + 3) & ~(int64_t)3);
  const unsigned bytes = (unsigned)(te - ts) * 4u;
  mbar_arrive_expect_tx(bar, bytes);
  bulk_load(buf, p.x + ts, bytes, bar);
  if (++c.tile == c.it.tiles) {
    c.item += gridDim.x;
    c.tile = 0;
    if (c.item < p.items) c.it = plane_item<P>(p, c.item);
  }
}

// a - b saturated to +-2^30: an item bound relative to a tile (far outside
// when it lies in another tile).
__device__ __forceinline__ int rel_sat(int64_t a, int64_t b) {
  constexpr int64_t kFar = int64_t(1) << 30;
  return (int)max(min(a - b, kFar), -kFar);
}

// ---------------------------------------------------------------------------
// The scan of one tile in shared memory, shared by both kernels.
// ---------------------------------------------------------------------------

// One thread's share of a tile between the two phases.
template <int P>
struct RunState {
  float v[kRunOf<P>];     // my run in scan order: inputs, then running values, then outputs
  float pre[P];      // class totals of my floats before the head
  float ex[P];       // segmented totals of the lanes before mine in the warp
  int hp;            // the head: scan position in my run where a plane starts (kRunOf<P>: none)
  bool head_before;  // a lane before mine in the warp holds a head
  // Planes no longer than a run (several boundaries in it): the position of
  // my first float (in scan order) within its plane, the last head, and the
  // item-relative plane of my first float.
  int pos0, hlast, qfirst;
};

// Planes of L <= kRunOf<P> floats (every run holds a boundary): the head
// (first plane start in scan order), the last one, my first float's position
// in its plane and, forward, the item-relative plane it lies in.  rr is my
// run's first float relative to the item's start (> -kPlaneAlign), magic is
// ceil(2^32 / L); every dividend stays below 2^32 / L.
template <int P, bool REV>
__device__ __forceinline__ void find_heads_short(int rr, int L, unsigned long long magic, RunState<P>& st) {
  constexpr int R = kRunOf<P>;
  const unsigned u = (unsigned)(rr + (REV ? R - 1 : 0) + 64 * L);  // > 0: 64 L exceeds any negative rr
  const int q = (int)(((unsigned long long)u * magic) >> 32);
  st.pos0 = (int)u - q * L;
  st.qfirst = q - 64;
  const int first = REV ? (st.pos0 + 1 == L ? 0 : st.pos0 + 1) : (st.pos0 == 0 ? 0 : L - st.pos0);
  st.hp = first;
  st.hlast = first + L * (int)(((unsigned long long)(unsigned)(R - 1 - first) * magic) >> 32);
}

// The head of my run (first float at a in the tile) and, for a reduction,
// dd: my floats before the end of plane q - 1 of the item (1..kRunOf<P>), else -1.
// Forward: boundaries at lo + q*L, q = 0 .. planes (the one at hi splits a
// reduction's last run); reverse: a plane starts (in scan order) at its last
// float, lo + q*L - 1, q >= 1.  Boundaries past the item only split floats
// that are never stored.  rlo, rhi: the item's bounds relative to the tile.
// one_plane: the item is one plane (boundaries at lo and hi only); else the
// item's planes, shorter than a tile, all lie in this one (0 <= rlo <
// kPlaneAlign) and Li, magic give L and ceil(2^32 / L).
template <int P, bool REV>
__device__ __forceinline__ void find_head(int a, int rlo, int rhi, bool one_plane, int Li, unsigned long long magic,
                                          int& hp, int& dd, int& q) {
  hp = kRunOf<P>;
  dd = -1;
  q = 0;
  if (one_plane) {
    if constexpr (!REV) {
      const int d1 = rlo - a, d2 = rhi - a;
      if (d1 >= 0 && d1 < kRunOf<P>) hp = d1;
      else if (d2 >= 0 && d2 < kRunOf<P>) hp = d2;
      if (d2 >= 1 && d2 <= kRunOf<P>) {
        dd = d2;
        q = 1;
      }
    } else {
      const int e = a + kRunOf<P> - rhi;
      if (e >= 0 && e < kRunOf<P>) hp = e;
    }
  } else {
    const int rr = a - rlo;
    if constexpr (!REV) {
      q = rr <= 0 ? 0 : (int)(((unsigned long long)(rr - 1) * magic) >> 32) + 1;
      const int d = q * Li - rr;  // >= 0
      if (d < kRunOf<P>) hp = d;
      if (d >= 1 && d <= kRunOf<P>) dd = d;
    } else {
      const int g = rr + kRunOf<P>;  // > 0
      const int qr = (int)(((unsigned long long)g * magic) >> 32);
      const int e = g - qr * Li;
      if (qr >= 1 && e < kRunOf<P>) hp = e;
    }
  }
}

// Phase 1: read my run (memory order reversed for a reverse scan), scan it
// per class, then the warp's segmented scan of the run totals; lane 31
// writes the warp's last-segment totals and head flag.  st.hp must be set.
template <int P, bool SCAN, bool REV, bool EXCL, typename Op, bool MULTI = false>
__device__ __forceinline__ void runs_phase1(RunState<P>& st, const float* buf, int a, float (&wagg)[kNW][P],
                                            int (&wflag)[kNW], int L = 0) {
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int hp = st.hp;
  {
    const float4* src = reinterpret_cast<const float4*>(buf + a);
#pragma unroll
    for (int k = 0; k < kChunksOf<P>; ++k) {
      const float4 q = src[k];
      const float e4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = 4 * k + c;
        st.v[REV ? kRunOf<P> - 1 - i : i] = SCAN ? e4[c] : Op::prep(e4[c]);
      }
    }
  }
  // 1. Sequential per-class scan of the run.  acc[c] runs over class c; the
  // first float of each class at or after the head starts it again.  v[e]
  // becomes the float's running value (inclusive, or the value before it
  // when exclusive); pre[c] ends as class c's total before the head.
  float acc[P];
#pragma unroll
  for (int c = 0; c < P; ++c) acc[c] = st.pre[c] = Op::identity();
  if constexpr (MULTI) {
    // Planes no longer than a run: a float restarts its class when it lies
    // in its plane's first row in scan order (position < P forward, >= L - P
    // reverse); the position walks with the float.  A reduction keeps every
    // running value.
    int pos = st.pos0;
#pragma unroll
    for (int e = 0; e < kRunOf<P>; ++e) {
      const int c = e % P;
      const bool restart = REV ? pos >= L - P : pos < P;
      const float before = restart ? Op::identity() : acc[c];
      acc[c] = restart ? st.v[e] : Op::combine(acc[c], st.v[e]);
      if constexpr (SCAN) st.v[e] = EXCL ? before : acc[c];
      else st.v[e] = acc[c];
      if constexpr (REV) pos = pos == 0 ? L - 1 : pos - 1;
      else pos = pos + 1 == L ? 0 : pos + 1;
    }
    // A class with no float after the last head keeps nothing for the new
    // plane (class c first appears hlast + ((c - hlast) mod P) floats in).
    const int hl = st.hlast;
#pragma unroll
    for (int c = 0; c < P; ++c)
      if (hl + ((c - hl % P + P) % P) >= kRunOf<P>) acc[c] = Op::identity();
  } else if (!__any_sync(kFullMask, hp > 0 && hp < kRunOf<P>)) {
    // No head inside a run of this warp (hp is 0 or kRunOf<P> everywhere).
#pragma unroll
    for (int e = 0; e < kRunOf<P>; ++e) {
      const int c = e % P;
      const float before = acc[c];
      acc[c] = Op::combine(acc[c], st.v[e]);
      if constexpr (SCAN) st.v[e] = EXCL ? before : acc[c];
    }
    if (hp == kRunOf<P>) {
#pragma unroll
      for (int c = 0; c < P; ++c) st.pre[c] = acc[c];
    }
  } else {
#pragma unroll
    for (int e = 0; e < kRunOf<P>; ++e) {
      const int c = e % P;
      const bool restart = (unsigned)(e - hp) < (unsigned)P;  // first of its class in the new plane
      const float before = restart ? Op::identity() : acc[c];
      acc[c] = restart ? st.v[e] : Op::combine(acc[c], st.v[e]);
      if constexpr (SCAN) st.v[e] = EXCL ? before : acc[c];
      if (e < hp) st.pre[c] = acc[c];
    }
    // A class with no float after a head near the run's end (positions
    // kRunOf<P> - P + c hold class c) keeps nothing for the new plane.
#pragma unroll
    for (int c = 0; c < P; ++c)
      if (kRunOf<P> - P + c < hp && hp < kRunOf<P>) acc[c] = Op::identity();
  }
  // 2. Segmented inclusive scan of the runs' last-segment totals across the
  // warp: lane l adds only lanes at or after hh, its last lane with a head
  // (every lane between hh and l has the same hh, so the Hillis-Steele steps
  // stay inside the segment).
  // (Planes no longer than a run: every lane holds a head, so lane l takes
  // only its own last segment and the steps are skipped.)
  const unsigned hmask = MULTI ? kFullMask : __ballot_sync(kFullMask, hp < kRunOf<P>);
  const unsigned upto = hmask & (kFullMask >> (31 - lane));
  const int hh = upto ? 31 - __clz((int)upto) : 0;
#pragma unroll
  for (int o = 1; o < (MULTI ? 1 : 32); o <<= 1) {
    const bool take = lane - o >= hh;
#pragma unroll
    for (int c = 0; c < P; ++c) {
      const float u = __shfl_up_sync(kFullMask, acc[c], o);
      if (take) acc[c] = Op::combine(u, acc[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < P; ++c) st.ex[c] = __shfl_up_sync(kFullMask, acc[c], 1);
  st.head_before = (hmask & ((1u << lane) - 1u)) != 0;
  if (lane == 31) {
#pragma unroll
    for (int c = 0; c < P; ++c) wagg[w][c] = acc[c];
    wflag[w] = hmask != 0;
  }
}

// Phase 2, after a barrier that published the warps' totals: cl gets the
// carry into my run's floats before its head, from `carry` (into the tile)
// and the warps before mine in order (a warp with a head restarts it); a
// scan adds it to those floats.  With `next` set, the last warp's lane 0
// writes there the carry out of the tile.
template <int P, bool SCAN, typename Op>
__device__ __forceinline__ void runs_phase2(RunState<P>& st, const float (&carry)[P], const float (&wagg)[kNW][P],
                                            const int (&wflag)[kNW], float* next, float (&cl)[P]) {
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  float cw[P];
#pragma unroll
  for (int c = 0; c < P; ++c) cw[c] = carry[c];
#pragma unroll
  for (int q = 0; q < kNW - 1; ++q) {
    if (q < w) {
      const bool f = wflag[q] != 0;
#pragma unroll
      for (int c = 0; c < P; ++c) cw[c] = f ? wagg[q][c] : Op::combine(cw[c], wagg[q][c]);
    }
  }
  if (next != nullptr && w == kNW - 1 && lane == 0) {
    const bool f = wflag[kNW - 1] != 0;
#pragma unroll
    for (int c = 0; c < P; ++c) next[c] = f ? wagg[kNW - 1][c] : Op::combine(cw[c], wagg[kNW - 1][c]);
  }
#pragma unroll
  for (int c = 0; c < P; ++c)
    cl[c] = lane == 0 ? cw[c] : (st.head_before ? st.ex[c] : Op::combine(cw[c], st.ex[c]));
  if constexpr (SCAN) {
#pragma unroll
    for (int e = 0; e < kRunOf<P>; ++e)
      if (e < st.hp) st.v[e] = Op::combine(cl[e % P], st.v[e]);
  }
}

// A scan's run back to its place in the tile (memory order).
template <int P, bool REV>
__device__ __forceinline__ void put_run(const float (&v)[kRunOf<P>], float* buf, int a) {
  float4* dst = reinterpret_cast<float4*>(buf + a);
#pragma unroll
  for (int k = 0; k < kChunksOf<P>; ++k) {
    float e4[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = 4 * k + c;
      e4[c] = v[REV ? kRunOf<P> - 1 - i : i];
    }
    dst[k] = make_float4(e4[0], e4[1], e4[2], e4[3]);
  }
}

// The floats [lo, hi) of a tile (relative to its first float, clamped to
// the tile) from shared memory to yt: one bulk store of the whole 16-byte
// granules [ga, gb) (thread 0), plain stores of the partial granules at the
// two ends (threads 0-7).  After a barrier that follows every thread's
// writes into buf and its fence_proxy_async_smem.
__device__ __forceinline__ void store_tile_out(const float* buf, float* yt, int lo, int hi) {
  const int t = threadIdx.x;
  const int ga = (lo + 3) & ~3;
  const int gb = hi & ~3;
  if (t == 0 && ga < gb) bulk_store(yt + ga, buf + ga, (unsigned)(gb - ga) * 4u);
  if (t < 8) {
    const int f = t < 4 ? lo + t : max(gb, ga) + (t - 4);
    if (f < (t < 4 ? min(ga, hi) : hi)) st_stream1(yt + f, buf[f]);
  }
}

template <int P, bool SCAN, bool REV, bool EXCL, typename Op, bool MULTI>
__global__ void __launch_bounds__(kT, 4) k_planes(PlaneRunParams p) {
  pdl_begin();
  __shared__ __align__(128) float s_buf[kStages][kTileOf<P>];
  __shared__ __align__(8) unsigned long long s_bar[kStages];
  // By tile parity (a reduction has no second barrier per tile, so a fast
  // warp may write the next tile's entries while others read these):
  __shared__ float s_wagg[2][kNW][P];  // each warp's last-segment totals
  __shared__ int s_wflag[2][kNW];      // the warp holds a head
  __shared__ float s_carry[2][P];      // carry into the next tile
  __shared__ Cursor s_pc;              // the producer's cursor (thread 0 only)
  const int t = threadIdx.x;
  const int a = (REV ? kT - 1 - t : t) * kRunOf<P>;  // my run's first float in a tile
  const int Li = (int)min(p.N * P, (int64_t)INT32_MAX);

  int outstanding = 0;  // thread 0: copies issued and not yet consumed
  if (t == 0) {
    Cursor pc;
    pc.item = blockIdx.x;
    pc.tile = 0;
    if (pc.item < p.items) pc.it = plane_item<P>(p, pc.item);
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(&s_bar[s], 1);
    fence_mbar_init();
#pragma unroll
    for (int s = 0; s < kStages; ++s)
      if (pc.item < p.items) {
        issue_tile<P>(p, pc, REV, s_buf[s], &s_bar[s]);
        ++outstanding;
      }
    s_pc = pc;
  }
  __syncthreads();

  int stage = 0;         // stage of the current tile
  unsigned phase = 0;    // its barrier's phase parity
  int par = 0;           // tile parity (warp totals and carries)
  bool started = false;  // a tile has been consumed
  bool fail = false;
  for (int64_t item = blockIdx.x; item < p.items && !fail; item += gridDim.x) {
    const PlaneItem it = plane_item<P>(p, item);
    for (int j = 0; j < it.tiles; ++j) {
      const bool landed = mbar_wait_copy(&s_bar[stage], phase);
      const int64_t ts = tile_start<P>(it, j, REV);
      float* buf = s_buf[stage];
      const int rlo = rel_sat(it.lo, ts);
      const int rhi = rel_sat(it.hi, ts);
      RunState<P> st;
      int dd = -1, qf = 0;
      if constexpr (MULTI) find_heads_short<P, REV>(a - rlo, Li, p.magic, st);
      else find_head<P, REV>(a, rlo, rhi, p.k == 1, Li, p.magic, st.hp, dd, qf);
      runs_phase1<P, SCAN, REV, EXCL, Op, MULTI>(st, buf, a, s_wagg[par], s_wflag[par], Li);
      // A scan, and a reduction of planes no longer than a run, use the tile
      // buffer after barrier 1 (outputs, running values): the previous
      // tile's buffer is refilled then.  Other reductions are done with it.
      constexpr bool kReuse = SCAN || MULTI;
      if constexpr (!kReuse) fence_proxy_async_smem();  // the buffer is refilled after barrier 1
      if constexpr (!SCAN && MULTI) put_run<P, false>(st.v, buf, a);  // running values, my own slots
      // Barrier 1: warp totals visible; every thread is past its wait for
      // this tile and done with the previous tile's buffer.
      if (__syncthreads_or(!landed)) {
        fail = true;
        break;
      }
      if (t == 0) {
        --outstanding;
        if (s_pc.item < p.items && (!kReuse || started)) {
          // Refill: a scan's previous buffer (once its bulk store has read
          // it), a reduction's current one (its runs are in registers).
          const int rs = kReuse ? (stage + kStages - 1) % kStages : stage;
          if constexpr (SCAN) bulk_store_wait_read();
          Cursor pc = s_pc;
          issue_tile<P>(p, pc, REV, s_buf[rs], &s_bar[rs]);
          s_pc = pc;
          ++outstanding;
        }
      }
      float carry[P], cl[P];
#pragma unroll
      for (int c = 0; c < P; ++c) carry[c] = j == 0 ? Op::identity() : s_carry[par][c];
      runs_phase2<P, SCAN, Op>(st, carry, s_wagg[par], s_wflag[par], s_carry[par ^ 1], cl);
      if constexpr (SCAN) {
        // The item's floats in the tile leave by one bulk store.
        put_run<P, REV>(st.v, buf, a);
        fence_proxy_async_smem();
        __syncthreads();
        store_tile_out(buf, p.y + ts, min(max(rlo, 0), kTileOf<P>), min(max(rhi, 0), kTileOf<P>));
        fence_proxy_async_smem();
      } else if constexpr (MULTI) {
        // Every plane ending in my run (forward, at position L - 1: my
        // floats e1, e1 + L, ...): its class totals are the running values
        // at its last row, read back from my own slots of the tile, with my
        // carry for the plane that began before my run (a class whose last
        // float lies in an earlier run: the carry alone).
        const int L = Li;
        int q = st.qfirst;
        for (int e = L - 1 - st.pos0; e < kRunOf<P>; e += L, ++q) {
          if (q < 0 || q >= it.planes) continue;
          float* out = p.y + (it.first + q) * P;
#pragma unroll
          for (int c = 0; c < P; ++c) {
            const int idx = e - ((e % P - c + P) % P);  // class c's last float of this plane
            float val = cl[c];
            if (idx >= 0) {
              const float r = buf[a + idx];
              val = idx < st.hp ? Op::combine(cl[c], r) : r;
            }
            st_plain(out + c, finish(val, p.flags, p.N));
          }
        }
        fence_proxy_async_smem();  // the buffer is refilled after the next tile's barrier 1
      } else {
        // A plane ending in my run: its class totals are my carry plus my
        // floats before the boundary.
        if (dd >= 1 && qf >= 1 && qf <= it.planes) {
          float* out = p.y + (it.first + qf - 1) * P;
#pragma unroll
          for (int c = 0; c < P; ++c) st_plain(out + c, finish(Op::combine(cl[c], st.pre[c]), p.flags, p.N));
        }
      }
      started = true;
      par ^= 1;
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (t == 0) {
    if (fail) {
      // A copy that never landed (its bounded wait ran out): report it, and
      // let no copy of this block still write into its shared memory after
      // it leaves (bounded waits, the failed one first).
      atomicOr(p.err_word, 1u);
      for (int k = 0; k < outstanding; ++k) {
        mbar_wait_copy(&s_bar[stage], phase);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if constexpr (SCAN) bulk_store_wait_all();  // the stores read shared memory until done
  }
}

// ---------------------------------------------------------------------------
// Scans as column groups, any P of 3 .. 128 columns.
//
// A run of whole rows per thread (k_planes) leaves wide planes one or two
// rows a thread and the lane scan P classes.  Here thread t owns column
// group g = t % G (V = 4, 2 or 1 adjacent columns: G = P / V groups) of a
// run of S consecutive rows (S = 9, 17, 33 for V = 4, 2, 1), row group
// t / G (reversed for a reverse scan); the 128 / G row groups of a tile make
// it whole rows (threads past them idle, holding zeros).  A thread's classes
// are its V components in every row, so its scan is one addition per float
// and a plane boundary restarts all V at once.  The lanes of a warp with the
// same g (G apart) carry the row groups' totals in log2(32 / G) shuffle
// steps of a segmented scan; warps fold their per-group totals through
// shared memory, with a head flag per warp and group.  A tile's rows start
// anywhere in a 16-byte granule: it lands by one bulk copy of its whole
// granules, delta floats in, and leaves by one bulk store of its whole
// granules plus plain stores of the partial ones at its two ends.  S is 1
// modulo 32 / gcd(P, 32), so a warp's threads read consecutive V-float
// slots of every row of their runs: no bank conflicts.  Planes must be
// longer than a run (N > S rows: at most one boundary per run).
// ---------------------------------------------------------------------------
template <int V>
constexpr int kCgS = planes_cg_run_rows_v(V);
template <int V>
constexpr int kCgBuf = kT * kCgS<V> * V + (V == 4 ? 0 : 8);  // floats per stage: the largest tile (and, for
                                                            // float2 / float groups, its two partial granules)

template <int V>
__device__ __forceinline__ void cg_ld(const float* p, float (&o)[V]) {
  if constexpr (V == 4) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    o[0] = q.x;
    o[1] = q.y;
    o[2] = q.z;
    o[3] = q.w;
  } else if constexpr (V == 2) {
    const float2 q = *reinterpret_cast<const float2*>(p);
    o[0] = q.x;
    o[1] = q.y;
  } else {
    o[0] = *p;
  }
}
template <int V>
__device__ __forceinline__ void cg_st(float* p, const float (&o)[V]) {
  if constexpr (V == 4) *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  else if constexpr (V == 2) *reinterpret_cast<float2*>(p) = make_float2(o[0], o[1]);
  else *p = o[0];
}

// An item of k planes (tiles of TR whole rows from its first row).
__device__ __forceinline__ PlaneItem cg_item(const PlaneRunParams& p, int TR, int64_t i) {
  PlaneItem it;
  it.first = i * p.k;
  const int64_t planes = min(p.k, p.outer - it.first);
  it.planes = (int)planes;
  it.lo = it.first * p.N * p.P;
  it.hi = it.lo + planes * p.N * p.P;
  it.vlo = it.lo;
  it.tiles = (int)((planes * p.N + TR - 1) / TR);
  return it;
}

// Tile `c.tile` of the cursor's item (in scan order): its whole granules.
__device__ __forceinline__ void cg_issue(const PlaneRunParams& p, int TR, Cursor& c, bool rev, float* buf,
                                         unsigned long long* bar) {
  if (c.item >= p.items) return;
  const int64_t tr0 = (int64_t)(rev ? c.it.tiles - 1 - c.tile : c.tile) * TR;
  const int64_t f0 = c.it.lo + tr0 * p.P;
  const int64_t f1 = min(f0 + (int64_t)TR * p.P, c.it.hi);
  const int64_t a0 = f0 & ~(int64_t)3, a1 = (f1 + 3) & ~(int64_t)3;
  const unsigned bytes = (unsigned)(a1 - a0) * 4u;
  mbar_arrive_expect_tx(bar, bytes);
  bulk_load(buf, p.x + a0, bytes, bar);
  if (++c.tile == c.it.tiles) {
    c.item += gridDim.x;
    c.tile = 0;
    if (c.item < p.items) c.it = cg_item(p, TR, c.item);
  }
}

// GMAX: the most column groups the instance takes (8 or 32; shared memory
// for the warp totals).  GFIX: the group count when fixed at compile time
// (16 and 32 columns), else 0 (taken from p.P).
template <int V, int GMAX, int GFIX, bool REV, bool EXCL>
__global__ void __launch_bounds__(kT, 4) k_planes_cg(PlaneRunParams p) {
  pdl_begin();
  constexpr int S = kCgS<V>;
  __shared__ __align__(128) float s_buf[kStages][kCgBuf<V>];
  __shared__ __align__(8) unsigned long long s_bar[kStages];
  __shared__ float s_wagg[2][kNW][GMAX * V];  // each warp's last-segment totals, by column group
  __shared__ unsigned char s_wflag[2][kNW][GMAX];  // a head in the warp's lanes of the group
  __shared__ float s_carry[2][GMAX * V];
  __shared__ Cursor s_pc;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int w = t >> 5;
  const int P = GFIX ? GFIX * V : p.P;
  const int G = GFIX ? GFIX : P / V;
  const int RG = kT / G;  // row groups per tile
  const int TR = RG * S;  // rows per tile
  const int g = t % G;
  const bool active = (GFIX && kT % GFIX == 0) || t / G < RG;  // row groups fill the block with 4 or 8 groups
  const int m = REV ? RG - 1 - t / G : t / G;  // my row group, in memory order (idle: out of range)
  const int row0 = m * S;                       // its first row in a tile
  const unsigned gmask = __match_any_sync(kFullMask, g);  // lanes of my column group
  const int glead = __ffs(gmask) - 1;                     // the first of them
  const int Ni = (int)min(p.N, (int64_t)INT32_MAX);

  int outstanding = 0;
  if (t == 0) {
    Cursor pc;
    pc.item = blockIdx.x;
    pc.tile = 0;
    if (pc.item < p.items) pc.it = cg_item(p, TR, pc.item);
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(&s_bar[s], 1);
    fence_mbar_init();
#pragma unroll
    for (int s = 0; s < kStages; ++s)
      if (pc.item < p.items) {
        cg_issue(p, TR, pc, REV, s_buf[s], &s_bar[s]);
        ++outstanding;
      }
    s_pc = pc;
  }
  __syncthreads();

  int stage = 0;
  unsigned phase = 0;
  int par = 0;
  bool started = false;
  bool fail = false;
  for (int64_t item = blockIdx.x; item < p.items && !fail; item += gridDim.x) {
    const PlaneItem it = cg_item(p, TR, item);
    const int64_t item_rows = (int64_t)it.planes * p.N;
    for (int j = 0; j < it.tiles; ++j) {
      const bool landed = mbar_wait_copy(&s_bar[stage], phase);
      const int jt = REV ? it.tiles - 1 - j : j;  // memory tile index
      const int64_t tr0 = (int64_t)jt * TR;       // its first row (item-relative)
      const int64_t f0 = it.lo + tr0 * P;         // its first float
      const int delta = V == 4 ? 0 : (int)(f0 & 3);  // where it lies in the copied granules
      const int rows = (int)min((int64_t)TR, item_rows - tr0);
      float* buf = s_buf[stage];
      // The head: forward, the first plane start at or after my first row
      // (rows q*N, q = 0 .. planes; the one at the item's end isolates rows
      // past it); reverse, the last row of a plane (q*N - 1, q >= 1).
      const int rr = (int)min(tr0 + row0, (int64_t)INT32_MAX / 2);  // my first row, item-relative
      int hp = S;
      if (active) {
        if (p.k == 1) {
          if constexpr (!REV) {
            const int d = rr == 0 ? 0 : Ni - rr;
            if (d >= 0 && d < S) hp = d;
          } else {
            const int e = rr + S - Ni;
            if (e >= 0 && e < S) hp = e;
          }
        } else {
          if constexpr (!REV) {
            const int q = rr == 0 ? 0 : (int)(((unsigned long long)(rr - 1) * p.magic) >> 32) + 1;
            const int d = q * Ni - rr;
            if (d < S) hp = d;
          } else {
            const int gq = rr + S;
            const int q = (int)(((unsigned long long)gq * p.magic) >> 32);
            const int e = gq - q * Ni;
            if (q >= 1 && e < S) hp = e;
          }
        }
      }
      // 1. My rows in scan order, scanned per component; the head row
      // restarts all V.
      const float* src = buf + delta + row0 * P + V * g;
      float v[S][V];
#pragma unroll
      for (int e = 0; e < S; ++e) {
        if (active) {
          cg_ld<V>(src + (REV ? S - 1 - e : e) * P, v[e]);
        } else {
#pragma unroll
          for (int c = 0; c < V; ++c) v[e][c] = 0.f;
        }
      }
      float acc[V];
#pragma unroll
      for (int c = 0; c < V; ++c) acc[c] = 0.f;
#pragma unroll
      for (int e = 0; e < S; ++e) {
        const bool restart = e == hp;
#pragma unroll
        for (int c = 0; c < V; ++c) {
          const float before = restart ? 0.f : acc[c];
          acc[c] = before + v[e][c];
          v[e][c] = EXCL ? before : acc[c];
        }
      }
      // 2. Segmented scan over the row groups of my column group in this
      // warp (lanes G apart): lane l adds lanes at or after its last lane
      // with a head.
      const unsigned hmask = __ballot_sync(kFullMask, hp < S) & gmask;
      const unsigned upto = hmask & (kFullMask >> (31 - lane));
      const int hh = upto ? 31 - __clz((int)upto) : glead;
      float inc[V];
#pragma unroll
      for (int c = 0; c < V; ++c) inc[c] = acc[c];
      for (int o = G; o < 32; o <<= 1) {
        float u[V];
#pragma unroll
        for (int c = 0; c < V; ++c) u[c] = __shfl_up_sync(kFullMask, inc[c], o);
        if (lane - o >= hh) {
#pragma unroll
          for (int c = 0; c < V; ++c) inc[c] = u[c] + inc[c];
        }
      }
      float ex[V];
#pragma unroll
      for (int c = 0; c < V; ++c) ex[c] = __shfl_up_sync(kFullMask, inc[c], G);
      const bool head_before = (hmask & ((1u << lane) - 1u)) != 0;
      if (lane >= 32 - G) {  // the last lane of my group in this warp holds its totals
#pragma unroll
        for (int c = 0; c < V; ++c) s_wagg[par][w][g * V + c] = inc[c];
        s_wflag[par][w][g] = hmask != 0;
      }
      if (__syncthreads_or(!landed)) {
        fail = true;
        break;
      }
      if (t == 0) {
        --outstanding;
        if (s_pc.item < p.items && started) {
          const int rs = (stage + kStages - 1) % kStages;
          bulk_store_wait_read();
          Cursor pc = s_pc;
          cg_issue(p, TR, pc, REV, s_buf[rs], &s_bar[rs]);
          s_pc = pc;
          ++outstanding;
        }
      }
      // 3. Carry into my warp for my column group, then into my row group.
      float cw[V];
#pragma unroll
      for (int c = 0; c < V; ++c) cw[c] = j == 0 ? 0.f : s_carry[par][g * V + c];
#pragma unroll
      for (int q = 0; q < kNW - 1; ++q) {
        if (q < w) {
          const bool restart = s_wflag[par][q][g] != 0;
#pragma unroll
          for (int c = 0; c < V; ++c) {
            const float a = s_wagg[par][q][g * V + c];
            cw[c] = restart ? a : cw[c] + a;
          }
        }
      }
      if (w == kNW - 1 && lane >= 32 - G) {
        const bool restart = s_wflag[par][kNW - 1][g] != 0;
#pragma unroll
        for (int c = 0; c < V; ++c) {
          const float a = s_wagg[par][kNW - 1][g * V + c];
          s_carry[par ^ 1][g * V + c] = restart ? a : cw[c] + a;
        }
      }
      float cl[V];
#pragma unroll
      for (int c = 0; c < V; ++c) cl[c] = lane < G ? cw[c] : (head_before ? ex[c] : cw[c] + ex[c]);
      // 4. Rows before the head take the carry; back in place, then the
      // tile's rows leave: whole granules by one bulk store, the partial
      // ones at its ends by plain stores.
      if (active) {
        float* dst = buf + delta + row0 * P + V * g;
#pragma unroll
        for (int e = 0; e < S; ++e) {
          if (e < hp) {
#pragma unroll
            for (int c = 0; c < V; ++c) v[e][c] = cl[c] + v[e][c];
          }
          cg_st<V>(dst + (REV ? S - 1 - e : e) * P, v[e]);
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      store_tile_out(buf, p.y + (f0 - delta), delta, delta + rows * P);
      fence_proxy_async_smem();
      started = true;
      par ^= 1;
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (t == 0) {
    if (fail) {
      atomicOr(p.err_word, 1u);
      for (int k = 0; k < outstanding; ++k) {
        mbar_wait_copy(&s_bar[stage], phase);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    bulk_store_wait_all();
  }
}


// Reductions as column groups (9 .. 128 columns): the same tiles, groups and
// runs as the scans, walked forward.  A thread keeps the combination of its
// rows before its head (pre) and from it on; the segmented lane scan and
// the warp fold carry the runs' last segments as for a scan.  The plane that
// ends in a thread's run (at most one: N > S) gets that thread's carry
// combined with its pre, V columns written by the thread.  A tile's rows go
// to registers before the tile's one barrier, after which its buffer is
// refilled at once; the warp totals alternate by tile parity.
// ---------------------------------------------------------------------------
template <int V, int GMAX, int GFIX, typename Op>
__global__ void __launch_bounds__(kT, 4) k_planes_cg_reduce(PlaneRunParams p) {
  pdl_begin();
  constexpr int S = kCgS<V>;
  __shared__ __align__(128) float s_buf[kStages][kCgBuf<V>];
  __shared__ __align__(8) unsigned long long s_bar[kStages];
  __shared__ float s_wagg[2][kNW][GMAX * V];
  __shared__ unsigned char s_wflag[2][kNW][GMAX];
  __shared__ float s_carry[2][GMAX * V];
  __shared__ Cursor s_pc;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int w = t >> 5;
  const int P = GFIX ? GFIX * V : p.P;
  const int G = GFIX ? GFIX : P / V;
  const int RG = kT / G;
  const int TR = RG * S;
  const int g = t % G;
  const bool active = (GFIX && kT % GFIX == 0) || t / G < RG;
  const int row0 = (t / G) * S;
  const unsigned gmask = __match_any_sync(kFullMask, g);
  const int glead = __ffs(gmask) - 1;
  const int Ni = (int)min(p.N, (int64_t)INT32_MAX);

  int outstanding = 0;
  if (t == 0) {
    Cursor pc;
    pc.item = blockIdx.x;
    pc.tile = 0;
    if (pc.item < p.items) pc.it = cg_item(p, TR, pc.item);
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(&s_bar[s], 1);
    fence_mbar_init();
#pragma unroll
    for (int s = 0; s < kStages; ++s)
      if (pc.item < p.items) {
        cg_issue(p, TR, pc, false, s_buf[s], &s_bar[s]);
        ++outstanding;
      }
    s_pc = pc;
  }
  __syncthreads();

  int stage = 0;
  unsigned phase = 0;
  int par = 0;
  bool fail = false;
  for (int64_t item = blockIdx.x; item < p.items && !fail; item += gridDim.x) {
    const PlaneItem it = cg_item(p, TR, item);
    for (int j = 0; j < it.tiles; ++j) {
      const bool landed = mbar_wait_copy(&s_bar[stage], phase);
      const int64_t tr0 = (int64_t)j * TR;
      const int64_t f0 = it.lo + tr0 * P;
      const int delta = V == 4 ? 0 : (int)(f0 & 3);
      const float* buf = s_buf[stage];
      // The head (the first plane start at or after my first row) and the
      // plane that ends in my run: its last row is dd - 1 rows in, and it is
      // plane qf - 1 of the item.
      const int rr = (int)min(tr0 + row0, (int64_t)INT32_MAX / 2);
      int hp = S, dd = 0, qf = 0;
      if (active) {
        if (p.k == 1) {
          const int d = rr == 0 ? 0 : Ni - rr;
          if (d >= 0 && d < S) hp = d;
          if (rr > 0 && d >= 1 && d <= S) {
            dd = d;
            qf = 1;
          }
        } else {
          const int q = rr == 0 ? 0 : (int)(((unsigned long long)(rr - 1) * p.magic) >> 32) + 1;
          const int d = q * Ni - rr;
          if (d < S) hp = d;
          if (q >= 1 && d >= 1 && d <= S) {
            dd = d;
            qf = q;
          }
        }
      }
      // 1. My rows combined per component, before the head and from it on.
      float pre[V], post[V];
#pragma unroll
      for (int c = 0; c < V; ++c) pre[c] = post[c] = Op::identity();
      if (active) {
        const float* src = buf + delta + row0 * P + V * g;
#pragma unroll
        for (int e = 0; e < S; ++e) {
          float r[V];
          cg_ld<V>(src + e * P, r);
#pragma unroll
          for (int c = 0; c < V; ++c) {
            const float x = Op::prep(r[c]);
            if (e < hp) pre[c] = Op::combine(pre[c], x);
            else post[c] = Op::combine(post[c], x);
          }
        }
      }
      fence_proxy_async_smem();  // the buffer is refilled after the barrier
      // 2. Segmented scan of the runs' last segments over my column group's
      // lanes in this warp.
      const unsigned hmask = __ballot_sync(kFullMask, hp < S) & gmask;
      const unsigned upto = hmask & (kFullMask >> (31 - lane));
      const int hh = upto ? 31 - __clz((int)upto) : glead;
      float inc[V];
#pragma unroll
      for (int c = 0; c < V; ++c) inc[c] = hp < S ? post[c] : pre[c];
      for (int o = G; o < 32; o <<= 1) {
        float u[V];
#pragma unroll
        for (int c = 0; c < V; ++c) u[c] = __shfl_up_sync(kFullMask, inc[c], o);
        if (lane - o >= hh) {
#pragma unroll
          for (int c = 0; c < V; ++c) inc[c] = Op::combine(u[c], inc[c]);
        }
      }
      float ex[V];
#pragma unroll
      for (int c = 0; c < V; ++c) ex[c] = __shfl_up_sync(kFullMask, inc[c], G);
      const bool head_before = (hmask & ((1u << lane) - 1u)) != 0;
      if (lane >= 32 - G) {
#pragma unroll
        for (int c = 0; c < V; ++c) s_wagg[par][w][g * V + c] = inc[c];
        s_wflag[par][w][g] = hmask != 0;
      }
      // The one barrier: warp totals visible, every thread done with the
      // tile's buffer, which is refilled now.
      if (__syncthreads_or(!landed)) {
        fail = true;
        break;
      }
      if (t == 0) {
        --outstanding;
        if (s_pc.item < p.items) {
          Cursor pc = s_pc;
          cg_issue(p, TR, pc, false, s_buf[stage], &s_bar[stage]);
          s_pc = pc;
          ++outstanding;
        }
      }
      // 3. Carry into my warp for my column group, then into my run.
      float cw[V];
#pragma unroll
      for (int c = 0; c < V; ++c) cw[c] = j == 0 ? Op::identity() : s_carry[par][g * V + c];
#pragma unroll
      for (int q = 0; q < kNW - 1; ++q) {
        if (q < w) {
          const bool restart = s_wflag[par][q][g] != 0;
#pragma unroll
          for (int c = 0; c < V; ++c) {
            const float a = s_wagg[par][q][g * V + c];
            cw[c] = restart ? a : Op::combine(cw[c], a);
          }
        }
      }
      if (w == kNW - 1 && lane >= 32 - G) {
        const bool restart = s_wflag[par][kNW - 1][g] != 0;
#pragma unroll
        for (int c = 0; c < V; ++c) {
          const float a = s_wagg[par][kNW - 1][g * V + c];
          s_carry[par ^ 1][g * V + c] = restart ? a : Op::combine(cw[c], a);
        }
      }
      // 4. The plane ending in my run: the carry and my rows before its end.
      if (dd >= 1 && qf <= it.planes) {
        float* out = p.y + (it.first + qf - 1) * P + V * g;
#pragma unroll
        for (int c = 0; c < V; ++c) {
          const float cl = lane < G ? cw[c] : (head_before ? ex[c] : Op::combine(cw[c], ex[c]));
          st_plain(out + c, finish(Op::combine(cl, pre[c]), p.flags, p.N));
        }
      }
      par ^= 1;
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (t == 0 && fail) {
    atomicOr(p.err_word, 1u);
    for (int k = 0; k < outstanding; ++k) {
      mbar_wait_copy(&s_bar[stage], phase);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Few long planes: one tile per block, the carry by look-back.
//
// The block with ticket t (tickets in scan order, plane after plane)
//   1. starts bulk copies of tile t and of tile u = t - lag (the second
//      normally served from L2: u was first read lag tiles ago);
//   2. writes out tile u: its carry is the sum of the tiles before it in its
//      plane, read from the 32-ary look-back tree (warp L reads level L;
//      every node it needs was published about lag tickets ago), then the
//      tile scan of both kernels with that carry, and a bulk store;
//   3. sums tile t per class (a fixed tree) and publishes the sums, and every
//      parent node this tile completes, as the row look-back does.
// Steps 2 and 3 interleave: the loads of tile u's look-back nodes go out
// before the wait for tile t, whose node word goes out as soon as its sums
// are in (no wait of tile u's delays it), then tile u's scan and bulk store,
// and last the parents tile t completes.
// Tickets are taken in order by running blocks
// and a block waits only on tiles of smaller tickets, so every wait ends;
// each is bounded all the same.  (A persistent form, each block taking its
// next ticket and starting its copies while it works on the current one, ran
// at a third of this speed: the ticket's round trip and the wait for the
// previous store's shared-memory reads stalled the whole block every tile.)
// ---------------------------------------------------------------------------
template <int P>
struct LbTile {
  int64_t plane, j;  // plane and scan-order tile index
  int64_t lo, hi;    // the plane's floats
  int64_t ts;        // the tile's first float
  bool real;         // the plane has tile j
};

// Tickets are below 2^31 (the host bounds them by the node words).
template <int P, bool REV>
__device__ __forceinline__ LbTile<P> lb_tile(const PlaneLbParams& p, int64_t q) {
  const int64_t L = p.N * P;
  LbTile<P> g;
  g.plane = (unsigned)q / (unsigned)p.tiles;
  g.j = q - g.plane * p.tiles;
  g.lo = g.plane * L;
  g.hi = g.lo + L;
  const int64_t vlo = g.lo - g.lo % kPlaneAlign<P>;
  const int64_t nt = (g.hi - vlo + kTileOf<P> - 1) / kTileOf<P>;
  g.real = g.j < nt;
  g.ts = vlo + (REV ? nt - 1 - g.j : g.j) * kTileOf<P>;
  return g;
}

template <int P>
__device__ __forceinline__ void lb_copy(const PlaneLbParams& p, const LbTile<P>& g, float* buf,
                                        unsigned long long* bar) {
  const int64_t te = min(g.ts + kTileOf<P>, (g.hi + 3) & ~(int64_t)3);
  const unsigned bytes = (unsigned)(te - g.ts) * 4u;
  mbar_arrive_expect_tx(bar, bytes);
  bulk_load(buf, p.x + g.ts, bytes, bar);
}

template <int P, bool REV, bool EXCL>
__global__ void __launch_bounds__(kT, kLbBlocks) k_planes_lb(PlaneLbParams p) {
  pdl_begin();
  __shared__ __align__(128) float s_new[kTileOf<P>];  // tile `ticket`
  __shared__ __align__(128) float s_old[kTileOf<P>];  // tile `ticket - lag`
  __shared__ __align__(8) unsigned long long s_bar[2];
  __shared__ float s_wagg[kNW][P];
  __shared__ int s_wflag[kNW];
  __shared__ float s_red[kNW][P];
  __shared__ float s_part[kPlanesLbLevels][P];
  __shared__ unsigned s_ticket, s_epoch;
  __shared__ int s_fail, s_copies;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int w = t >> 5;
  const unsigned* abort_word = p.err_word + 1;
  const int64_t total = p.outer * p.tiles;
  const int a = (REV ? kT - 1 - t : t) * kRunOf<P>;  // my run's first float in a tile

  if (t == 0) {
    const Ticket tk = take_ticket(p.ticket_word);
    s_ticket = tk.ticket;
    s_epoch = tk.epoch;
    s_fail = 0;
    // Every other ticket is taken before the last one: reset for the next launch.
    if ((int64_t)tk.ticket == total + p.lag - 1) next_launch(p.ticket_word, tk.epoch);
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    fence_mbar_init();
    int copies = 0;
    if ((int64_t)tk.ticket < total) {
      const LbTile<P> g = lb_tile<P, REV>(p, tk.ticket);
      if (g.real) {
        lb_copy<P>(p, g, s_new, &s_bar[0]);
        copies |= 1;
      }
    }
    const int64_t u = (int64_t)tk.ticket - p.lag;
    if (u >= 0 && u < total) {
      const LbTile<P> g = lb_tile<P, REV>(p, u);
      if (g.real) {
        lb_copy<P>(p, g, s_old, &s_bar[1]);
        copies |= 2;
      }
    }
    s_copies = copies;
  }
  __syncthreads();
  const int64_t ticket = s_ticket;
  const unsigned epoch = s_epoch;
  if (ticket >= total + p.lag) {  // a stale counter: no copy was started, touch nothing
    if (t == 0) atomicOr(p.err_word, 2u);
    return;
  }
  int levels = 1;
  while (levels < kPlanesLbLevels && ((p.tiles - 1) >> (5 * levels)) != 0) ++levels;

  const int64_t u = ticket - p.lag;
  const bool pub = ticket < total;  // tile `ticket` is summed and published
  const LbTile<P> gt = lb_tile<P, REV>(p, pub ? ticket : 0);
  const LbTile<P> gu = lb_tile<P, REV>(p, u >= 0 ? u : 0);
  const bool wr = u >= 0 && gu.real;  // tile u is written out

  // 1. The loads of tile u's look-back nodes go out first (warp L reads
  // level L; every node it needs was published about lag tickets ago), so
  // that their latency passes while tile `ticket` is on its way from HBM.
  const unsigned long long* node = nullptr;  // my lane's node, if any
  unsigned long long word[P];
  if (wr && w < levels) {
    int64_t off = 0, count = p.tiles;
    for (int q = 0; q < w; ++q) {
      off += count;
      count >>= 5;
    }
    const int64_t m = gu.j >> (5 * w);
    const int d = (int)(m & 31);
    if (lane < d) {
      node = p.node_val + gu.plane * 2 * p.tiles * P + (off + (m - d) + lane) * P;
      load_node_classes<P>(node, word);
    }
  }

  // 2. Tile `ticket`'s class sums: my run's, in scan order (the classes as
  // the tile scan numbers them), only the plane's own floats; warp trees,
  // then the warp sums in order; warp 0 publishes them at once.
  float own[P];
#pragma unroll
  for (int c = 0; c < P; ++c) own[c] = 0.f;
  bool landed = true;
  if (pub && gt.real) {  // an empty last tile publishes zeros
    landed = mbar_wait_copy(&s_bar[0], 0u);
    const int tlo = rel_sat(gt.lo, gt.ts);
    const int thi = rel_sat(gt.hi, gt.ts);
    const float4* src = reinterpret_cast<const float4*>(s_new + a);
    const bool edge = tlo > a || thi < a + kRunOf<P>;
#pragma unroll
    for (int k = 0; k < kChunksOf<P>; ++k) {
      const float4 q = src[k];
      const float e4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = 4 * k + c;  // memory position a + i
        const int e = REV ? kRunOf<P> - 1 - i : i;
        const bool in = !edge || (a + i >= tlo && a + i < thi);
        own[e % P] += in ? e4[c] : 0.f;
      }
    }
#pragma unroll
    for (int c = 0; c < P; ++c) {
      own[c] = warp_reduce<OpSum>(own[c]);
      if (lane == 0) s_red[w][c] = own[c];
    }
  }
  // A copy that never landed: nothing published (the tiles behind wait out
  // and fail) and no outputs.
  const auto give_up = [&]() {
    if (t == 0) {
      atomicOr(p.err_word, 1u);
      atomicExch(p.err_word + 1, epoch);
      if (s_copies & 1) mbar_wait_copy(&s_bar[0], 0u);
      if (s_copies & 2) mbar_wait_copy(&s_bar[1], 0u);
    }
  };
  if (__syncthreads_or(!landed)) {
    give_up();
    return;
  }
  unsigned long long* tvals = p.node_val + gt.plane * 2 * p.tiles * P;
  const bool publishing = pub && ticket != p.stall_tile;
  if (pub && gt.real) {
#pragma unroll
    for (int c = 0; c < P; ++c) {
      float r = s_red[0][c];
#pragma unroll
      for (int q = 1; q < kNW; ++q) r += s_red[q][c];
      own[c] = r;
    }
  }
  if (publishing && w == 0 && lane < P) st_relaxed_u64(tvals + gt.j * P + lane, pack_node(epoch, pick_class<P>(own, lane)));

  // 3. Tile u up to its block fold: the look-back partials (the words not
  // yet published are polled, bounded), then the run and lane scans of the
  // reread (normally an L2 hit).
  RunState<P> st;
  int rlo = 0, rhi = 0;
  landed = true;
  if (wr) {
    if (w < levels) {
      bool fail = false;
      float sib[P];
#pragma unroll
      for (int c = 0; c < P; ++c) sib[c] = 0.f;
      if (node) settle_node_classes<P>(node, word, epoch, p.spin_limit, abort_word, &fail, sib);
#pragma unroll
      for (int c = 0; c < P; ++c) {
        const float part = warp_tree_adjacent(sib[c]);
        if (lane == 0) s_part[w][c] = part;
      }
      if (__any_sync(kFullMask, fail) && lane == 0) s_fail = 1;
    }
    landed = mbar_wait_copy(&s_bar[1], 0u);
    rlo = rel_sat(gu.lo, gu.ts);
    rhi = rel_sat(gu.hi, gu.ts);
    int dd, qf;
    find_head<P, REV>(a, rlo, rhi, true, 0, 0ull, st.hp, dd, qf);
    runs_phase1<P, true, REV, EXCL, OpSum>(st, s_old, a, s_wagg, s_wflag);
  }
  // The barrier publishes s_part and the warp folds.
  if (__syncthreads_or(!landed)) {
    give_up();
    return;
  }

  // 4. The rest of tile u: each class's carry is its look-back partials from
  // the lowest level up; back in place, then one bulk store.
  if (wr) {
    float carry[P], cl[P];
#pragma unroll
    for (int c = 0; c < P; ++c) {
      float e = 0.f;
      for (int L = 0; L < levels; ++L) e += s_part[L][c];
      carry[c] = e;
    }
    runs_phase2<P, true, OpSum>(st, carry, s_wagg, s_wflag, nullptr, cl);
    put_run<P, REV>(st.v, s_old, a);
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (wr) store_tile_out(s_old, p.y + gu.ts, min(max(rlo, 0), kTileOf<P>), min(max(rhi, 0), kTileOf<P>));

  // 5. Every parent node tile `ticket` completes (warp 0, after the store is
  // on its way): the 31 siblings before it and its own sums.
  if (publishing && w == 0 && (gt.j & 31) == 31) {
    bool fail = false;
    int64_t off = 0, count = p.tiles, m = gt.j;
    for (int L = 0; L < levels && (m & 31) == 31; ++L) {
      float sib[P];
#pragma unroll
      for (int c = 0; c < P; ++c) sib[c] = 0.f;
      if (lane < 31)
        wait_node_classes<P>(tvals + (off + (m - 31) + lane) * P, epoch, p.spin_limit, abort_word, &fail, sib);
      if (__any_sync(kFullMask, fail)) break;
#pragma unroll
      for (int c = 0; c < P; ++c) {
        const float parent = warp_tree_adjacent(lane < 31 ? sib[c] : own[c]);
        own[c] = __shfl_sync(kFullMask, parent, 0);
      }
      const int64_t next_off = off + count;
      if (lane < P)
        st_relaxed_u64(tvals + (next_off + (m >> 5)) * P + lane, pack_node(epoch, pick_class<P>(own, lane)));
      off = next_off;
      count >>= 5;
      m >>= 5;
    }
    if (fail && lane == 0) s_fail = 1;
  }
  // s_fail's other writers came before the barriers above; thread 0 wrote
  // the last one itself.
  if (t == 0) {
    if (s_fail) {
      atomicOr(p.err_word, 1u);
      atomicExch(p.err_word + 1, epoch);
    }
    // Both copies have landed (waited above); the bulk store must have read
    // this block's shared memory before the block leaves.  Its writes need
    // no wait: they are complete when the grid is.
    bulk_store_wait_read();
  }
}

// ---------------------------------------------------------------------------
// Few long planes as column groups (6 .. 128 columns): one tile per block,
// each column's carry by look-back.
//
// The tiles, groups and runs of k_planes_cg over one plane each (tiles of TR
// whole rows from the plane's start, in scan order), with the tickets and
// the per-plane 32-ary look-back tree of k_planes_lb: P node words per tile,
// one per column.  The block with ticket t
//   1. copies tile t and rereads tile u = t - lag (normally an L2 hit);
//   2. sums tile t per column -- each thread its run, a tree over the lanes
//      of its column group, then the warps in order -- and publishes the P
//      words at once;
//   3. reads tile u's look-back, level by level: warp w takes siblings w,
//      w + 4, ... with lane = column (lanes cover columns 32 apart), the
//      warps' partials added in warp order, the levels lowest first;
//   4. scans tile u as k_planes_cg does, that carry entering its first
//      warp, and bulk-stores it;
//   5. publishes every parent tile t completes (its 31 siblings as the
//      look-back reads them, then its own sums).
// Every wait is on a smaller ticket and bounded; every sum has a fixed order.
// ---------------------------------------------------------------------------
// One warp's share of a level's siblings for one column: siblings w, w + 4,
// ... below d of the node row at `first` (sibling s at first + s * P), all
// loads issued before any is waited on (bounded), summed in sibling order.
__device__ __forceinline__ float cg_lb_siblings(const unsigned long long* first, int P, int d, int w, unsigned epoch,
                                                int64_t limit, const unsigned* abort_word, bool* fail) {
  constexpr int kPer = (31 + kNW - 1) / kNW;
  unsigned long long word[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int sb = w + kNW * i;
    word[i] = sb < d ? ld_relaxed_u64(first + (int64_t)sb * P) : 0ull;
  }
  float part = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int sb = w + kNW * i;
    if (sb < d)
      part += (unsigned)(word[i] >> 32) == epoch ? __uint_as_float((unsigned)word[i])
                                                 : wait_node(first + (int64_t)sb * P, epoch, limit, abort_word, fail);
  }
  return part;
}

template <int V, int GMAX, int GFIX, bool REV, bool EXCL>
__global__ void __launch_bounds__(kT, 6) k_planes_cg_lb(PlaneLbParams p) {
  pdl_begin();
  constexpr int S = kCgS<V>;
  constexpr int PMAX = GMAX * V;  // the most columns the instance takes
  __shared__ __align__(128) float s_new[kCgBuf<V>];  // tile `ticket`
  __shared__ __align__(128) float s_old[kCgBuf<V>];  // tile `ticket - lag`
  __shared__ __align__(8) unsigned long long s_bar[2];
  // Per-warp partials: tile sums, then look-back sums, then (step 4, after
  // the look-back's last barrier) the warps' scan totals.
  __shared__ float s_part[kNW][PMAX];
  float(&s_wagg)[kNW][PMAX] = s_part;
  __shared__ unsigned char s_wflag[kNW][GMAX];
  __shared__ float s_carry[PMAX];  // carry into tile u, per column
  __shared__ float s_own[PMAX];    // tile `ticket`'s sums, per column
  __shared__ unsigned s_ticket, s_epoch;
  __shared__ int s_fail, s_copies;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int w = t >> 5;
  const unsigned* abort_word = p.err_word + 1;
  const int P = GFIX ? GFIX * V : p.P;
  const int G = GFIX ? GFIX : P / V;
  const int RG = kT / G;
  const int TR = RG * S;
  const int g = t % G;
  const bool active = (GFIX && kT % GFIX == 0) || t / G < RG;
  const int m = REV ? RG - 1 - t / G : t / G;
  const int row0 = m * S;
  const unsigned gmask = __match_any_sync(kFullMask, g);
  const int glead = __ffs(gmask) - 1;
  const int64_t total = p.outer * p.tiles;
  const int64_t L = p.N * P;  // floats per plane
  const int Ni = (int)min(p.N, (int64_t)INT32_MAX);

  // A ticket's plane and its tile in memory order (scan-order tile j).
  const auto locate = [&](int64_t q, int64_t& plane, int64_t& j, int64_t& tr0, int& rows) {
    plane = (unsigned)q / (unsigned)p.tiles;
    j = q - plane * p.tiles;
    const int64_t jt = REV ? p.tiles - 1 - j : j;
    tr0 = jt * TR;
    rows = (int)min((int64_t)TR, p.N - tr0);
  };
  const auto copy = [&](int64_t q, float* buf, unsigned long long* bar) {
    int64_t plane, j, tr0;
    int rows;
    locate(q, plane, j, tr0, rows);
    const int64_t f0 = plane * L + tr0 * P;
    const int64_t a0 = f0 & ~(int64_t)3, a1 = (f0 + (int64_t)rows * P + 3) & ~(int64_t)3;
    const unsigned bytes = (unsigned)(a1 - a0) * 4u;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load(buf, p.x + a0, bytes, bar);
  };

  if (t == 0) {
    const Ticket tk = take_ticket(p.ticket_word);
    s_ticket = tk.ticket;
    s_epoch = tk.epoch;
    s_fail = 0;
    if ((int64_t)tk.ticket == total + p.lag - 1) next_launch(p.ticket_word, tk.epoch);
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    fence_mbar_init();
    int copies = 0;
    if ((int64_t)tk.ticket < total) {
      copy(tk.ticket, s_new, &s_bar[0]);
      copies |= 1;
    }
    const int64_t u = (int64_t)tk.ticket - p.lag;
    if (u >= 0 && u < total) {
      copy(u, s_old, &s_bar[1]);
      copies |= 2;
    }
    s_copies = copies;
  }
  __syncthreads();
  const int64_t ticket = s_ticket;
  const unsigned epoch = s_epoch;
  if (ticket >= total + p.lag) {  // a stale counter: no copy was started, touch nothing
    if (t == 0) atomicOr(p.err_word, 2u);
    return;
  }
  int levels = 1;
  while (levels < kPlanesLbLevels && ((p.tiles - 1) >> (5 * levels)) != 0) ++levels;
  const int64_t u = ticket - p.lag;
  const bool pub = ticket < total;
  const bool wr = u >= 0;
  const auto give_up = [&]() {
    if (t == 0) {
      atomicOr(p.err_word, 1u);
      atomicExch(p.err_word + 1, epoch);
      if (s_copies & 1) mbar_wait_copy(&s_bar[0], 0u);
      if (s_copies & 2) mbar_wait_copy(&s_bar[1], 0u);
    }
  };

  // 2. Tile `ticket`'s column sums (only the plane's rows), published at once.
  int64_t tplane = 0, tj = 0, ttr0 = 0;
  int trows = 0;
  bool landed = true;
  if (pub) {
    locate(ticket, tplane, tj, ttr0, trows);
    landed = mbar_wait_copy(&s_bar[0], 0u);
    const int delta = V == 4 ? 0 : (int)((tplane * L + ttr0 * P) & 3);
    float a[V];
#pragma unroll
    for (int c = 0; c < V; ++c) a[c] = 0.f;
    if (active) {
      const float* src = s_new + delta + row0 * P + V * g;
#pragma unroll
      for (int e = 0; e < S; ++e) {
        if (row0 + e < trows) {
          float r[V];
          cg_ld<V>(src + e * P, r);
#pragma unroll
          for (int c = 0; c < V; ++c) a[c] += r[c];
        }
      }
    }
    // A tree over the lanes of my column group in this warp (lane + o in
    // range only), its first lane holding the warp's sums.
    for (int o = G; o < 32; o <<= 1) {
#pragma unroll
      for (int c = 0; c < V; ++c) {
        const float q = __shfl_down_sync(kFullMask, a[c], o);
        if (lane + o < 32) a[c] += q;
      }
    }
    if (lane < G) {
#pragma unroll
      for (int c = 0; c < V; ++c) s_part[w][g * V + c] = a[c];
    }
  }
  if (__syncthreads_or(!landed)) {
    give_up();
    return;
  }
  const bool publishing = pub && ticket != p.stall_tile;
  unsigned long long* tvals = p.node_val + tplane * 2 * p.tiles * P;
  if (pub) {
    for (int c = t; c < P; c += kT) {
      float r = s_part[0][c];
#pragma unroll
      for (int q = 1; q < kNW; ++q) r += s_part[q][c];
      s_own[c] = r;
      if (publishing) st_relaxed_u64(tvals + tj * P + c, pack_node(epoch, r));
    }
  }
  __syncthreads();  // s_part free again; s_own complete

  // 3. Tile u's carry, per column: the look-back, level by level.
  int64_t uplane = 0, uj = 0, utr0 = 0;
  int urows = 0;
  if (wr) {
    locate(u, uplane, uj, utr0, urows);
    const unsigned long long* uvals = p.node_val + uplane * 2 * p.tiles * P;
    for (int c = t; c < P; c += kT) s_carry[c] = 0.f;
    int64_t off = 0, count = p.tiles;
    for (int Lv = 0; Lv < levels; ++Lv) {
      const int64_t mm = uj >> (5 * Lv);
      const int d = (int)(mm & 31);
      bool fail = false;
      for (int c = lane; c < P; c += 32) s_part[w][c] = cg_lb_siblings(uvals + (off + (mm - d)) * P + c, P, d, w, epoch, p.spin_limit, abort_word, &fail);
      if (__any_sync(kFullMask, fail) && lane == 0) s_fail = 1;
      __syncthreads();
      for (int c = t; c < P; c += kT) {
        float r = s_part[0][c];
#pragma unroll
        for (int q = 1; q < kNW; ++q) r += s_part[q][c];
        s_carry[c] += r;
      }
      __syncthreads();
      off += count;
      count >>= 5;
    }
  }

  // 4. Tile u: the scan of k_planes_cg with that carry.
  landed = true;
  float v[S][V];
  int hp = S;
  int delta_u = 0;
  if (wr) {
    landed = mbar_wait_copy(&s_bar[1], 0u);
    delta_u = V == 4 ? 0 : (int)((uplane * L + utr0 * P) & 3);
    const int rr = (int)min(utr0 + row0, (int64_t)INT32_MAX / 2);
    if (active) {
      if constexpr (!REV) {
        const int dh = rr == 0 ? 0 : Ni - rr;
        if (dh >= 0 && dh < S) hp = dh;
      } else {
        const int e = rr + S - Ni;
        if (e >= 0 && e < S) hp = e;
      }
    }
    const float* src = s_old + delta_u + row0 * P + V * g;
#pragma unroll
    for (int e = 0; e < S; ++e) {
      if (active) {
        cg_ld<V>(src + (REV ? S - 1 - e : e) * P, v[e]);
      } else {
#pragma unroll
        for (int c = 0; c < V; ++c) v[e][c] = 0.f;
      }
    }
  }
  float acc[V];
#pragma unroll
  for (int c = 0; c < V; ++c) acc[c] = 0.f;
  if (wr) {
#pragma unroll
    for (int e = 0; e < S; ++e) {
      const bool restart = e == hp;
#pragma unroll
      for (int c = 0; c < V; ++c) {
        const float before = restart ? 0.f : acc[c];
        acc[c] = before + v[e][c];
        v[e][c] = EXCL ? before : acc[c];
      }
    }
  }
  const unsigned hmask = __ballot_sync(kFullMask, hp < S) & gmask;
  const unsigned upto = hmask & (kFullMask >> (31 - lane));
  const int hh = upto ? 31 - __clz((int)upto) : glead;
  float inc[V];
#pragma unroll
  for (int c = 0; c < V; ++c) inc[c] = acc[c];
  for (int o = G; o < 32; o <<= 1) {
    float q[V];
#pragma unroll
    for (int c = 0; c < V; ++c) q[c] = __shfl_up_sync(kFullMask, inc[c], o);
    if (lane - o >= hh) {
#pragma unroll
      for (int c = 0; c < V; ++c) inc[c] = q[c] + inc[c];
    }
  }
  float ex[V];
#pragma unroll
  for (int c = 0; c < V; ++c) ex[c] = __shfl_up_sync(kFullMask, inc[c], G);
  const bool head_before = (hmask & ((1u << lane) - 1u)) != 0;
  if (lane >= 32 - G) {
#pragma unroll
    for (int c = 0; c < V; ++c) s_wagg[w][g * V + c] = inc[c];
    s_wflag[w][g] = hmask != 0;
  }
  if (__syncthreads_or(!landed)) {
    give_up();
    return;
  }
  if (wr) {
    float cw[V];
#pragma unroll
    for (int c = 0; c < V; ++c) cw[c] = s_carry[g * V + c];
#pragma unroll
    for (int q = 0; q < kNW - 1; ++q) {
      if (q < w) {
        const bool restart = s_wflag[q][g] != 0;
#pragma unroll
        for (int c = 0; c < V; ++c) {
          const float a = s_wagg[q][g * V + c];
          cw[c] = restart ? a : cw[c] + a;
        }
      }
    }
    float cl[V];
#pragma unroll
    for (int c = 0; c < V; ++c) cl[c] = lane < G ? cw[c] : (head_before ? ex[c] : cw[c] + ex[c]);
    if (active) {
      float* dst = s_old + delta_u + row0 * P + V * g;
#pragma unroll
      for (int e = 0; e < S; ++e) {
        if (e < hp) {
#pragma unroll
          for (int c = 0; c < V; ++c) v[e][c] = cl[c] + v[e][c];
        }
        cg_st<V>(dst + (REV ? S - 1 - e : e) * P, v[e]);
      }
    }
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (wr) store_tile_out(s_old, p.y + (uplane * L + utr0 * P - delta_u), delta_u, delta_u + urows * P);

  // 5. Every parent tile `ticket` completes: its 31 siblings (warp
  // partials in warp order, as the look-back), then its own sums.
  if (publishing && (tj & 31) == 31) {
    bool fail = false;
    int64_t off = 0, count = p.tiles, mm = tj;
    for (int Lv = 0; Lv + 1 < levels && (mm & 31) == 31; ++Lv) {
      const int64_t next_off = off + count;
      for (int c = lane; c < P; c += 32)
        s_part[w][c] = cg_lb_siblings(tvals + (off + (mm - 31)) * P + c, P, 31, w, epoch, p.spin_limit, abort_word, &fail);
      __syncthreads();
      for (int c = t; c < P; c += kT) {
        float r = s_part[0][c];
#pragma unroll
        for (int q = 1; q < kNW; ++q) r += s_part[q][c];
        r += s_own[c];
        s_own[c] = r;
        st_relaxed_u64(tvals + (next_off + (mm >> 5)) * P + c, pack_node(epoch, r));
      }
      __syncthreads();
      off = next_off;
      count >>= 5;
      mm >>= 5;
    }
    if (fail) s_fail = 1;
  }
  __syncthreads();
  if (t == 0) {
    if (s_fail) {
      atomicOr(p.err_word, 1u);
      atomicExch(p.err_word + 1, epoch);
    }
    bulk_store_wait_read();
  }
}

template <typename K>
int occupancy_of(K kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kT, 0) != cudaSuccess) return 0;
  return n;
}

}  // namespace
}  // namespace lr
