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

      // 1. Suffix of each thread's VEC items, right to left.
      float inc[SUB], exc[SUB];
#pragma unroll
      for (int s = 0; s < SUB; ++s) {
#pragma unroll
        for (int i = VEC - 2; i >= 0; --i) cur[s][i] += cur[s][i + 1];
        // 2. Inclusive suffix over lanes: lane l gets the sum over lanes >= l.
        float v = cur[s][0];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float u = __shfl_down_sync(kFullMask, v, o);
          if (lane + o < 32) v += u;
        }
        inc[s] = v;
        const float e = __shfl_down_sync(kFullMask, v, 1);
        exc[s] = (lane == 31) ? 0.f : e;
        if (lane == 0) sh_w[par][s][w] = v;  // the warp's total
      }
      __syncthreads();

      // 3. Warp totals -> exclusive suffix over warps, sub-tile totals.
      float stot[SUB], wexc[SUB];
#pragma unroll
      for (int s = 0; s < SUB; ++s) {
        float wt[kNW];
#pragma unroll
        for (int q = 0; q < kNW; ++q) wt[q] = sh_w[par][s][q];
        stot[s] = tree_sum<kNW>(wt);
        float acc = 0.f;
#pragma unroll
        for (int q = kNW - 1; q >= 1; --q)
          if (q > w) acc += wt[q];
        wexc[s] = acc;
      }
      // 4. Sub-tiles to the right inside this tile.
      float rs[SUB];
      rs[SUB - 1] = 0.f;
#pragma unroll
      for (int s = SUB - 2; s >= 0; --s) rs[s] = stot[s + 1] + rs[s + 1];
      const float tile_total = stot[0] + rs[0];
      const float carry = carry_hi + carry_lo;

      // 5. Offsets, outputs.
#pragma unroll
      for (int s = 0; s < SUB; ++s) {
        const float off = exc[s] + (wexc[s] + (rs[s] + carry));
#pragma unroll
        for (int i = 0; i < VEC; ++i) cur[s][i] += off;
      }
      store_tile<VEC, SUB>(cur, yr, base, N, t);

      // 6. Blocked carry: fold every kCarryFold tiles to keep chains short.
      carry_lo += tile_total;
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

int occupancy_rscan_rows(int variant) {
  switch (variant) {
    case kRScanV1S4: return occupancy_of(k_rscan_rows<1, 4>);
    case kRScanV4S2: return occupancy_of(k_rscan_rows<4, 2>);
    case kRScanV4S4: return occupancy_of(k_rscan_rows<4, 4>);
    default: return 0;
  }
}

}  // namespace lr
