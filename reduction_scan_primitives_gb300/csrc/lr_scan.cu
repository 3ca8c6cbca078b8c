// lr_scan.cu -- reverse inclusive cumulative sum along rows (sm_103a).
//
// y[i, j] = x[i, j] + x[i, j+1] + ... + x[i, N-1]   (POPCORNBENCH trace l1_p91,
// problem statement: cumsum(x.flip(1), 1).flip(1) on a [32768, 32768] fp32
// array).
//
// One block owns a row and walks its tiles from right to left, carrying the
// sum of everything to the right in registers (the block-per-row, serial
// tiles with a carry plan of that trace).  Inside a tile each thread owns VEC
// consecutive elements in each of SUB sub-tiles, so a warp's loads and stores
// cover 32*VEC*4 contiguous bytes (the blocked, contiguous-per-thread layout
// the trace settles on after its strided layout double-counted).
//
// Every output is built from additions over its own suffix only:
//   thread-local suffix + (lane-exclusive suffix within the warp
//   + (warp-exclusive suffix within the sub-tile + (sub-tiles to the right
//   + carry))).
// The trace's formula tile_total - prefix_before(j) + carry is not used: it
// subtracts two large numbers to get a small one, which loses the accuracy
// the per-element tolerance (relative to that element's own suffix) asks for.
#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

constexpr int kNW = kThreads / 32;
constexpr int kCarryFold = 32;  // tiles per fold of the blocked carry

template <int VEC, int SUB>
__device__ __forceinline__ void load_tile(float (&v)[SUB][VEC], const float* xr, int64_t base,
                                          int64_t N, int t) {
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    const int64_t j = base + (int64_t)s * kThreads * VEC + (int64_t)t * VEC;
    if constexpr (VEC == 4) {
      // N % 4 == 0 on this path, so j < N means all four are in range.
      float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < N) q = ld_stream4(xr + j);
      v[s][0] = q.x;
      v[s][1] = q.y;
      v[s][2] = q.z;
      v[s][3] = q.w;
    } else {
      v[s][0] = (j < N) ? ld_stream1(xr + j) : 0.f;
    }
  }
}

template <int VEC, int SUB>
__device__ __forceinline__ void store_tile(const float (&v)[SUB][VEC], float* yr, int64_t base,
                                           int64_t N, int t) {
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    const int64_t j = base + (int64_t)s * kThreads * VEC + (int64_t)t * VEC;
    if (j < N) {
      if constexpr (VEC == 4) {
        st_stream4(yr + j, make_float4(v[s][0], v[s][1], v[s][2], v[s][3]));
      } else {
        st_stream1(yr + j, v[s][0]);
      }
    }
  }
}

// Suffix scan of one tile held in registers (v[s][i]: element s*256*VEC +
// t*VEC + i of the tile).  On return v holds each thread's local suffix, and
// for each sub-tile s the caller adds
//     exc[s] + (wexc[s] + (rs[s] + carry))
// where exc is the suffix over lanes to the right, wexc over warps to the
// right, rs over sub-tiles to the right, and carry over tiles to the right.
// `total` is the tile's sum (identical in every thread).  Contains one
// __syncthreads(); `sh` must not be written again until every thread of the
// block is past that barrier.
template <int VEC, int SUB>
struct TileScan {
  float exc[SUB], wexc[SUB], rs[SUB];
  float total;
};

template <int VEC, int SUB>
__device__ __forceinline__ TileScan<VEC, SUB> tile_suffix(float (&v)[SUB][VEC],
                                                         float (&sh)[SUB][kNW], int lane, int w) {
  TileScan<VEC, SUB> r;
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    // 1. Suffix of each thread's VEC items, right to left.
#pragma unroll
    for (int i = VEC - 2; i >= 0; --i) v[s][i] += v[s][i + 1];
    // 2. Inclusive suffix over lanes: lane l gets the sum over lanes >= l.
    float a = v[s][0];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_down_sync(kFullMask, a, o);
      if (lane + o < 32) a += u;
    }
    const float e = __shfl_down_sync(kFullMask, a, 1);
    r.exc[s] = (lane == 31) ? 0.f : e;
    if (lane == 0) sh[s][w] = a;  // the warp's total
  }
  __syncthreads();
  // 3. Warp totals -> exclusive suffix over warps, sub-tile totals.
  float stot[SUB];
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    float wt[kNW];
#pragma unroll
    for (int q = 0; q < kNW; ++q) wt[q] = sh[s][q];
    stot[s] = tree_sum<kNW>(wt);
    float acc = 0.f;
#pragma unroll
    for (int q = kNW - 1; q >= 1; --q)
      if (q > w) acc += wt[q];
    r.wexc[s] = acc;
  }
  // 4. Sub-tiles to the right inside this tile.
  r.rs[SUB - 1] = 0.f;
#pragma unroll
  for (int s = SUB - 2; s >= 0; --s) r.rs[s] = stot[s + 1] + r.rs[s + 1];
  r.total = stot[0] + r.rs[0];
  return r;
}

template <int VEC, int SUB>
__device__ __forceinline__ void add_offsets(float (&v)[SUB][VEC], const TileScan<VEC, SUB>& ts,
                                            float carry) {
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    const float off = ts.exc[s] + (ts.wexc[s] + (ts.rs[s] + carry));
#pragma unroll
    for (int i = 0; i < VEC; ++i) v[s][i] += off;
  }
}

// ---------------------------------------------------------------------------
// Block per row: tiles right to left, carry in registers, next tile
// prefetched into registers while the current one is scanned.
// ---------------------------------------------------------------------------
template <int VEC, int SUB>
__global__ void __launch_bounds__(kThreads) k_rscan_rows(RScanRowsParams p) {
  constexpr int64_t TILE = (int64_t)SUB * kThreads * VEC;
  __shared__ float sh_w[2][SUB][kNW];  // warp totals, double-buffered by tile parity
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int w = t >> 5;
  const int64_t N = p.N;
  const int64_t ntiles = (N + TILE - 1) / TILE;
  int par = 0;

  for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
    const float* xr = p.x + row * N;
    float* yr = p.y + row * N;
    float cur[SUB][VEC];
    float nxt[SUB][VEC];
    load_tile<VEC, SUB>(cur, xr, (ntiles - 1) * TILE, N, t);
    float carry_lo = 0.f, carry_hi = 0.f;
    int ncarry = 0;

    for (int64_t k = ntiles - 1; k >= 0; --k) {
      const int64_t base = k * TILE;
      if (k > 0) load_tile<VEC, SUB>(nxt, xr, base - TILE, N, t);  // prefetch the tile to the left
      const TileScan<VEC, SUB> ts = tile_suffix<VEC, SUB>(cur, sh_w[par], lane, w);
      add_offsets<VEC, SUB>(cur, ts, carry_hi + carry_lo);
      store_tile<VEC, SUB>(cur, yr, base, N, t);
      // Blocked carry: fold every kCarryFold tiles to keep chains short.
      carry_lo += ts.total;
      if (++ncarry == kCarryFold) {
        carry_hi += carry_lo;
        carry_lo = 0.f;
        ncarry = 0;
      }
      par ^= 1;
#pragma unroll
      for (int s = 0; s < SUB; ++s)
#pragma unroll
        for (int i = 0; i < VEC; ++i) cur[s][i] = nxt[s][i];
    }
  }
}

// ---------------------------------------------------------------------------
// Single-pass decoupled look-back, deterministic.
//
// Tiles of a row are numbered k = 0, 1, ... from the right end (scan order).
// A(k) is tile k's sum.  B(l, j) = A(j*2^l) + ... + A((j+1)*2^l - 1) is a
// dyadic block; B(0, k) = A(k), and B(l, j) = B(l-1, 2j) + B(l-1, 2j+1)
// (lower index first) is formed by whichever of its two children is
// published last, found with an exchange on an arrival word.  Tile k's
// exclusive suffix (everything to its right) is the sum, over the set bits l
// of k, of B(l, (k >> l) - 1): the binary decomposition of [0, k).  Which
// block values exist when a tile looks back depends on timing, but every
// value, and the way the tile combines them, does not, so the result is
// bit-identical from run to run.
//
// Forward progress: tickets are taken in scan order, so a tile only waits
// for tiles with smaller tickets, whose blocks are already running and never
// wait on later tiles.  Every wait is bounded; when one runs out the block
// records the failure (error word, plus this launch's epoch in the abort
// word so the other waiters stop early) and finishes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long pack_node(unsigned epoch, float v) {
  return ((unsigned long long)epoch << 32) | (unsigned long long)__float_as_uint(v);
}

__device__ __forceinline__ int64_t level_offset(int64_t tiles, int l) {
  int64_t off = 0;
  for (int q = 0; q < l; ++q) off += tiles >> q;
  return off;
}

// Poll a node until it carries this launch's epoch (or give up).
__device__ __forceinline__ float wait_node(const unsigned long long* node, unsigned epoch,
                                           int64_t limit, const unsigned* abort_word, bool* fail) {
  unsigned ns = 32;
  for (int64_t it = 0;; ++it) {
    const unsigned long long word = ld_acquire_u64(node);
    if ((unsigned)(word >> 32) == epoch) return __uint_as_float((unsigned)word);
    if (it >= limit || ld_relaxed_u32(abort_word) == epoch) {
      *fail = true;
      return 0.f;
    }
    __nanosleep(ns);
    if (ns < 1024) ns <<= 1;
  }
}

// Publish A(k) and complete every dyadic block this tile is the last child of.
__device__ void publish_up(unsigned long long* vals, unsigned* arrive, int64_t tiles, int64_t k,
                           float a, unsigned epoch, int64_t limit, const unsigned* abort_word,
                           bool* fail) {
  float val = a;
  int l = 0;
  int64_t j = k;
  int64_t off = 0;
  st_release_u64(vals + j, pack_node(epoch, val));
  while (true) {
    const int64_t pj = j >> 1;
    if (pj >= (tiles >> (l + 1))) break;  // the parent block runs past the row end
    const int64_t next_off = off + (tiles >> l);
    if (atom_exch_acq_rel(arrive + next_off + pj, epoch) != epoch) break;  // first child
    const float sib = wait_node(vals + off + (j ^ 1), epoch, limit, abort_word, fail);
    if (*fail) break;
    val = (j & 1) ? (sib + val) : (val + sib);
    ++l;
    j = pj;
    off = next_off;
    st_release_u64(vals + off + j, pack_node(epoch, val));
  }
}

template <int VEC, int SUB>
__global__ void __launch_bounds__(kThreads) k_rscan_lookback(RScanLookbackParams p) {
  constexpr int64_t TILE = (int64_t)SUB * kThreads * VEC;
  __shared__ float sh_w[SUB][kNW];
  __shared__ unsigned s_ticket;
  __shared__ float s_excl;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int w = t >> 5;
  const unsigned* abort_word = p.err_word + 1;

  if (t == 0) s_ticket = atomicAdd(p.tile_counter, 1u);
  __syncthreads();
  const int64_t ticket = s_ticket;
  const int64_t tiles = p.tiles_per_row;
  if (ticket >= p.rows * tiles) {  // a stale counter: touch nothing
    if (t == 0) atomicOr(p.err_word, 2u);
    return;
  }
  const int64_t row = ticket / tiles;
  const int64_t k = ticket - row * tiles;    // from the right
  const int64_t base = (tiles - 1 - k) * TILE;  // tiles are aligned at the row's left end
  const float* xr = p.x + row * p.N;
  float* yr = p.y + row * p.N;

  float v[SUB][VEC];
  load_tile<VEC, SUB>(v, xr, base, p.N, t);
  const TileScan<VEC, SUB> ts = tile_suffix<VEC, SUB>(v, sh_w, lane, w);

  if (w == 0) {
    unsigned long long* vals = p.node_val + row * 2 * tiles;
    unsigned* arrive = p.node_arrive + row * 2 * tiles;
    bool fail = false;
    if (lane == 0 && ticket != p.stall_tile)
      publish_up(vals, arrive, tiles, k, ts.total, p.epoch, p.spin_limit, abort_word, &fail);
    __syncwarp();
    float e = 0.f;
    if ((k >> lane) & 1) {
      const int64_t j = (k >> lane) - 1;
      e = wait_node(vals + level_offset(tiles, lane) + j, p.epoch, p.spin_limit, abort_word, &fail);
    }
    e = warp_sum(e);  // fixed tree over the decomposition's blocks
    const unsigned failed = __any_sync(kFullMask, fail);
    if (lane == 0) {
      s_excl = e;
      if (failed) {
        atomicOr(p.err_word, 1u);
        atomicExch(p.err_word + 1, p.epoch);
      }
    }
  }
  __syncthreads();
  add_offsets<VEC, SUB>(v, ts, s_excl);
  store_tile<VEC, SUB>(v, yr, base, p.N, t);
}

template <typename K>
int occupancy_of(K kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess) return 0;
  return n;
}

}  // namespace

cudaError_t launch_rscan_rows(int variant, const RScanRowsParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (variant) {
    case kRScanV1S4: k_rscan_rows<1, 4><<<g, kThreads, 0, s>>>(p); break;
    case kRScanV4S2: k_rscan_rows<4, 2><<<g, kThreads, 0, s>>>(p); break;
    case kRScanV4S4: k_rscan_rows<4, 4><<<g, kThreads, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

int64_t lookback_tile(int variant) {
  switch (variant) {
    case kLookbackV1: return 8 * kThreads * 1;
    case kLookbackV4: return 8 * kThreads * 4;
    default: return 0;
  }
}

cudaError_t launch_rscan_lookback(int variant, const RScanLookbackParams& p, int64_t grid,
                                  cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (variant) {
    case kLookbackV1: k_rscan_lookback<1, 8><<<g, kThreads, 0, s>>>(p); break;
    case kLookbackV4: k_rscan_lookback<4, 8><<<g, kThreads, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

int occupancy_rscan_lookback(int variant) {
  switch (variant) {
    case kLookbackV1: return occupancy_of(k_rscan_lookback<1, 8>);
    case kLookbackV4: return occupancy_of(k_rscan_lookback<4, 8>);
    default: return 0;
  }
}

int occupancy_rscan_rows(int variant) {
  switch (variant) {
    case kRScanV1S4: return occupancy_of(k_rscan_rows<1, 4>);
    case kRScanV4S2: return occupancy_of(k_rscan_rows<4, 2>);
    case kRScanV4S4: return occupancy_of(k_rscan_rows<4, 4>);
    default: return 0;
  }
}

}  // namespace lr
