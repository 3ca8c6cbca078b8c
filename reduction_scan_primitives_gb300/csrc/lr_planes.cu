// lr_planes.cu -- cumulative sums and reductions along the middle axis of
// [outer, N, P] for narrow planes of P = 2, 3 or 4 columns (sm_103a).
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
// to tile.  A tile of kPlanesTile floats lands in shared memory by one bulk
// copy (TMA engine), three tiles in flight per block; its start is the
// item's start rounded down to a 16-byte boundary (and to a multiple of P).
//
// Thread t of the 128 owns run m of kPlanesRun = 36 consecutive floats of the
// tile (m = t; m = 127 - t for a reverse scan, whose scan order runs down
// memory).  36 is a multiple of every P and every run starts at a multiple of
// P, so the column class of each of a thread's floats is known at compile
// time; as L > 36, a run holds at most one plane boundary (its "head": the
// scan position where a plane starts, in scan order).  A run is 9 float4
// chunks, an odd number, so the runs of 8 consecutive threads fall in
// distinct shared-memory banks.  The steps:
//   1. a sequential per-class scan over the run, restarting at the head;
//   2. a segmented shuffle scan of the run totals across the warp (per class,
//      the lanes before a lane's last head excluded);
//   3. the warps' totals through shared memory, folded in warp order with the
//      carry of the previous tile (same segment rule);
//   4. each float before its run's head gets its lane's carry; a scan writes
//      the run back in place and the tile leaves by one bulk store of its
//      whole 16-byte granules (the item's partial first and last granules by
//      plain stores); a reduction writes the P totals of each plane that ends
//      in the run.
// Every output is a sum over its own terms in a fixed order (an exclusive
// output leaves its own term out of the running value), nothing is
// subtracted, and reruns are bit-identical.  Floats of the tile outside the
// item (before its start, after its end) are loaded but fall in other
// segments, so they never reach an output; only the item's own floats are
// stored.
#include <algorithm>

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

constexpr int kT = kPlanesThreads;
constexpr int kNW = kT / 32;
constexpr int kRun = kPlanesRun;
constexpr int kTile = kPlanesTile;
constexpr int kChunks = kRun / 4;  // float4 chunks per run
constexpr int kStages = 3;
static_assert(kRun % 4 == 0 && kRun % 3 == 0 && (kChunks & 1) == 1,
              "runs hold whole float4 chunks, a multiple of every P, an odd number of chunks");
// Runs and tiles start on multiples of this many floats: 16 bytes and P.
template <int P>
constexpr int kPlaneAlign = P == 3 ? 12 : 4;

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
  it.tiles = (int)((it.hi - it.vlo + kTile - 1) / kTile);
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
__device__ __forceinline__ int64_t tile_start(const PlaneItem& it, int j, bool rev) {
  return it.vlo + (int64_t)(rev ? it.tiles - 1 - j : j) * kTile;
}

template <int P>
__device__ __forceinline__ void issue_tile(const PlaneRunParams& p, Cursor& c, bool rev, float* buf,
                                           unsigned long long* bar) {
  if (c.item >= p.items) return;
  const int64_t ts = tile_start(c.it, c.tile, rev);
  // Whole 16-byte granules up to the item's end: the last one lies in the
  // same page as the item's last float.
  const int64_t te = min(ts + kTile, (c.it.hi + 3) & ~(int64_t)3);
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

template <int P, bool SCAN, bool REV, bool EXCL, typename Op>
__global__ void __launch_bounds__(kT, 4) k_planes(PlaneRunParams p) {
  __shared__ __align__(128) float s_buf[kStages][kTile];
  __shared__ __align__(8) unsigned long long s_bar[kStages];
  // By tile parity (a reduction has no second barrier per tile, so a fast
  // warp may write the next tile's entries while others read these):
  __shared__ float s_wagg[2][kNW][P];  // each warp's last-segment totals
  __shared__ int s_wflag[2][kNW];      // the warp holds a head
  __shared__ float s_carry[2][P];      // carry into the next tile
  __shared__ Cursor s_pc;              // the producer's cursor (thread 0 only)
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int w = t >> 5;
  const int a = (REV ? kT - 1 - t : t) * kRun;  // my run's first float in a tile

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
      const int64_t ts = tile_start(it, j, REV);
      float* buf = s_buf[stage];

      // My run in scan order (memory order reversed for a reverse scan).
      float v[kRun];
      {
        const float4* src = reinterpret_cast<const float4*>(buf + a);
#pragma unroll
        for (int k = 0; k < kChunks; ++k) {
          const float4 q = src[k];
          const float e4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int i = 4 * k + c;
            v[REV ? kRun - 1 - i : i] = SCAN ? e4[c] : Op::prep(e4[c]);
          }
        }
      }
      if constexpr (!SCAN) fence_proxy_async_smem();  // the buffer is refilled after barrier 1

      // The head: the scan position in my run where a plane starts (kRun:
      // none).  Forward: boundaries at lo + q*L, q = 0 .. planes (the one at
      // hi splits a reduction's last run); reverse: a plane starts (in scan
      // order) at its last float, lo + q*L - 1, q >= 1.  Boundaries past the
      // item only split floats that are never stored.  For a reduction, dd
      // counts my floats before the end of plane first + qf - 1 (1..kRun),
      // or is -1.
      const int rlo = rel_sat(it.lo, ts);
      const int rhi = rel_sat(it.hi, ts);
      int hp = kRun, dd = -1, qf = 0;
      if (p.k == 1) {  // one plane: boundaries at lo and hi only
        if constexpr (!REV) {
          const int d1 = rlo - a, d2 = rhi - a;
          if (d1 >= 0 && d1 < kRun) hp = d1;
          else if (d2 >= 0 && d2 < kRun) hp = d2;
          if (d2 >= 1 && d2 <= kRun) {
            dd = d2;
            qf = 1;
          }
        } else {
          const int e = a + kRun - rhi;
          if (e >= 0 && e < kRun) hp = e;
        }
      } else {  // planes shorter than a tile, all in this one: 0 <= rlo < kPlaneAlign
        const int rr = a - rlo;
        const int Li = (int)(p.N * P);
        if constexpr (!REV) {
          qf = rr <= 0 ? 0 : (int)(((unsigned long long)(rr - 1) * p.magic) >> 32) + 1;
          const int d = qf * Li - rr;  // >= 0
          if (d < kRun) hp = d;
          if (d >= 1 && d <= kRun) dd = d;
        } else {
          const int g = rr + kRun;  // > 0
          const int qr = (int)(((unsigned long long)g * p.magic) >> 32);
          const int e = g - qr * Li;
          if (qr >= 1 && e < kRun) hp = e;
        }
      }

      // 1. Sequential per-class scan of the run.  acc[c] runs over class c;
      // the first float of each class at or after the head starts it again.
      // v[e] becomes the float's running value (inclusive, or the value
      // before it when exclusive); pre[c] ends as class c's total over the
      // floats before the head.
      float acc[P], pre[P];
#pragma unroll
      for (int c = 0; c < P; ++c) acc[c] = pre[c] = Op::identity();
      if (!__any_sync(kFullMask, hp > 0 && hp < kRun)) {
        // No head inside a run of this warp (hp is 0 or kRun everywhere).
#pragma unroll
        for (int e = 0; e < kRun; ++e) {
          const int c = e % P;
          const float before = acc[c];
          acc[c] = Op::combine(acc[c], v[e]);
          if constexpr (SCAN) v[e] = EXCL ? before : acc[c];
        }
        if (hp == kRun) {
#pragma unroll
          for (int c = 0; c < P; ++c) pre[c] = acc[c];
        }
      } else {
#pragma unroll
        for (int e = 0; e < kRun; ++e) {
          const int c = e % P;
          const bool restart = (unsigned)(e - hp) < (unsigned)P;  // first of its class in the new plane
          const float before = restart ? Op::identity() : acc[c];
          acc[c] = restart ? v[e] : Op::combine(acc[c], v[e]);
          if constexpr (SCAN) v[e] = EXCL ? before : acc[c];
          if (e < hp) pre[c] = acc[c];
        }
        // A class with no float after a head near the run's end (positions
        // kRun - P + c hold class c) keeps nothing for the new plane.
#pragma unroll
        for (int c = 0; c < P; ++c)
          if (kRun - P + c < hp && hp < kRun) acc[c] = Op::identity();
      }

      // 2. Segmented inclusive scan of the runs' last-segment totals across
      // the warp: lane l adds only lanes at or after hh, its last lane with a
      // head (every lane between hh and l has the same hh, so the
      // Hillis-Steele steps stay inside the segment).
      const unsigned hmask = __ballot_sync(kFullMask, hp < kRun);
      const unsigned upto = hmask & (kFullMask >> (31 - lane));
      const int hh = upto ? 31 - __clz((int)upto) : 0;
      float inc[P];
#pragma unroll
      for (int c = 0; c < P; ++c) inc[c] = acc[c];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const bool take = lane - o >= hh;
#pragma unroll
        for (int c = 0; c < P; ++c) {
          const float u = __shfl_up_sync(kFullMask, inc[c], o);
          if (take) inc[c] = Op::combine(u, inc[c]);
        }
      }
      float ex[P];  // the lanes before mine, within my first float's segment
#pragma unroll
      for (int c = 0; c < P; ++c) ex[c] = __shfl_up_sync(kFullMask, inc[c], 1);
      const bool head_before = (hmask & ((1u << lane) - 1u)) != 0;
      if (lane == 31) {
#pragma unroll
        for (int c = 0; c < P; ++c) s_wagg[par][w][c] = inc[c];
        s_wflag[par][w] = hmask != 0;
      }
      // Barrier 1: warp totals visible; every thread is past its wait for
      // this tile and done with the previous tile's buffer.
      if (__syncthreads_or(!landed)) {
        fail = true;
        break;
      }
      if (t == 0) {
        --outstanding;
        if (s_pc.item < p.items && (!SCAN || started)) {
          // Refill: a scan's previous buffer (once its bulk store has read
          // it), a reduction's current one (its runs are in registers).
          const int rs = SCAN ? (stage + kStages - 1) % kStages : stage;
          if constexpr (SCAN) bulk_store_wait_read();
          Cursor pc = s_pc;
          issue_tile<P>(p, pc, REV, s_buf[rs], &s_bar[rs]);
          s_pc = pc;
          ++outstanding;
        }
      }

      // 3. Carry into my warp: the previous tile's carry, then the warps
      // before mine in order (a warp with a head restarts it).
      float cw[P];
#pragma unroll
      for (int c = 0; c < P; ++c) cw[c] = j == 0 ? Op::identity() : s_carry[par][c];
#pragma unroll
      for (int q = 0; q < kNW - 1; ++q) {
        if (q < w) {
          const bool f = s_wflag[par][q] != 0;
#pragma unroll
          for (int c = 0; c < P; ++c) cw[c] = f ? s_wagg[par][q][c] : Op::combine(cw[c], s_wagg[par][q][c]);
        }
      }
      if (w == kNW - 1 && lane == 0) {
        const bool f = s_wflag[par][kNW - 1] != 0;
#pragma unroll
        for (int c = 0; c < P; ++c)
          s_carry[par ^ 1][c] = f ? s_wagg[par][kNW - 1][c] : Op::combine(cw[c], s_wagg[par][kNW - 1][c]);
      }
      float cl[P];  // carry into my run's floats before its head
#pragma unroll
      for (int c = 0; c < P; ++c)
        cl[c] = lane == 0 ? cw[c] : (head_before ? ex[c] : Op::combine(cw[c], ex[c]));

      if constexpr (SCAN) {
        // 4. Outputs: the floats before the head take the carry; the run
        // goes back to its place, and the item's floats in the tile leave by
        // one bulk store of their whole granules [ga, gb) plus plain stores
        // of the partial granules at the item's two ends.
#pragma unroll
        for (int e = 0; e < kRun; ++e)
          if (e < hp) v[e] = Op::combine(cl[e % P], v[e]);
        float4* dst = reinterpret_cast<float4*>(buf + a);
#pragma unroll
        for (int k = 0; k < kChunks; ++k) {
          float e4[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int i = 4 * k + c;
            e4[c] = v[REV ? kRun - 1 - i : i];
          }
          dst[k] = make_float4(e4[0], e4[1], e4[2], e4[3]);
        }
        fence_proxy_async_smem();
        __syncthreads();
        const int lo = min(max(rlo, 0), kTile);
        const int hi = min(max(rhi, 0), kTile);
        const int ga = (lo + 3) & ~3;
        const int gb = hi & ~3;
        float* yt = p.y + ts;
        if (t == 0 && ga < gb) bulk_store(yt + ga, buf + ga, (unsigned)(gb - ga) * 4u);
        if (t < 8) {
          const int f = t < 4 ? lo + t : max(gb, ga) + (t - 4);
          if (f < (t < 4 ? min(ga, hi) : hi)) st_stream1(yt + f, buf[f]);
        }
      }
      else {
        // 4. A plane ending in my run: its class totals are my carry plus my
        // floats before the boundary.
        if (dd >= 1 && qf >= 1 && qf <= it.planes) {
          float* out = p.y + (it.first + qf - 1) * P;
#pragma unroll
          for (int c = 0; c < P; ++c) st_plain(out + c, finish(Op::combine(cl[c], pre[c]), p.flags, p.N));
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

template <typename K>
int occupancy_of(K kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kT, 0) != cudaSuccess) return 0;
  return n;
}

template <int P, bool REV>
cudaError_t launch_scan_dir(const PlaneRunParams& p, dim3 g, cudaStream_t s) {
  if (p.flags & kScanExclusive) k_planes<P, true, REV, true, OpSum><<<g, kT, 0, s>>>(p);
  else k_planes<P, true, REV, false, OpSum><<<g, kT, 0, s>>>(p);
  return cudaGetLastError();
}

template <int P>
cudaError_t launch_scan_p(const PlaneRunParams& p, dim3 g, cudaStream_t s) {
  return (p.flags & kScanMirror) ? launch_scan_dir<P, false>(p, g, s) : launch_scan_dir<P, true>(p, g, s);
}

template <int P>
cudaError_t launch_reduce_p(int op, const PlaneRunParams& p, dim3 g, cudaStream_t s) {
  switch (op) {
    case kOpSum: k_planes<P, false, false, false, OpSum><<<g, kT, 0, s>>>(p); break;
    case kOpSumSq: k_planes<P, false, false, false, OpSumSq><<<g, kT, 0, s>>>(p); break;
    case kOpMax: k_planes<P, false, false, false, OpMax><<<g, kT, 0, s>>>(p); break;
    case kOpMin: k_planes<P, false, false, false, OpMin><<<g, kT, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <int P>
int occupancy_p(bool scan) {
  if (!scan) return occupancy_of(k_planes<P, false, false, false, OpSum>);
  return std::min({occupancy_of(k_planes<P, true, false, false, OpSum>),
                   occupancy_of(k_planes<P, true, false, true, OpSum>),
                   occupancy_of(k_planes<P, true, true, false, OpSum>),
                   occupancy_of(k_planes<P, true, true, true, OpSum>)});
}

}  // namespace

cudaError_t launch_planes_scan(int P, const PlaneRunParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (P) {
    case 2: return launch_scan_p<2>(p, g, s);
    case 3: return launch_scan_p<3>(p, g, s);
    case 4: return launch_scan_p<4>(p, g, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_planes_reduce(int P, int op, const PlaneRunParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (P) {
    case 2: return launch_reduce_p<2>(op, p, g, s);
    case 3: return launch_reduce_p<3>(op, p, g, s);
    case 4: return launch_reduce_p<4>(op, p, g, s);
    default: return cudaErrorInvalidValue;
  }
}

int occupancy_planes(int P, bool scan) {
  switch (P) {
    case 2: return occupancy_p<2>(scan);
    case 3: return occupancy_p<3>(scan);
    case 4: return occupancy_p<4>(scan);
    default: return 0;
  }
}

}  // namespace lr
