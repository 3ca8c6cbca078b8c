// lr_reduce.cu -- fp32 reduction kernels: 1D, rows (inner == 1) and strided
// axes (inner > 1), for sum, sum of squares, max and min (sm_103a).
//
// Design, by source:
//  * "High-Performance Reduction Kernels" README, 'Key design decisions':
//    float4 loads, warp-shuffle trees, one float per warp staged in shared
//    memory, an SM-aware grid, and a contiguous chunk per block.  Its
//    'Optimization: ILP4 accumulator' section: several independent loads in
//    flight per thread.  Here each thread issues U independent 128-bit loads
//    per step and sums them with a fixed tree.
//  * "Seven-step reduction: 30x from one kernel", V7: warp shuffle first, shared
//    memory only across warps.  Its atomicAdd(out, sum) finish is replaced by a
//    deterministic one: block partials go to scratch and the last block (found
//    with an integer ticket) adds them in index order, so reruns are
//    bit-identical.
//  * POPCORNBENCH trace l1_p47 (sum over dim=1 of [128, 4096, 4095]): threads
//    run across the contiguous inner dim (coalesced) and loop over the reduce
//    dim, several rows in flight; float4 columns only when inner % 4 == 0,
//    because an odd row stride breaks 16-byte alignment of later rows.
#include <algorithm>
#include <type_traits>

#include "lr_contig.cuh"
#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

// ---------------------------------------------------------------------------
// Short 1D arrays: one thread-block cluster, combined in distributed shared
// memory.  A short sum is bound by latency, not bandwidth: every load of the
// array is issued at once (one memory round trip), and the CTAs' results meet
// through the cluster's shared memory instead of a global ticket, so the
// launch pays no atomic and no second round trip through L2.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned cluster_ctarank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster: release this CTA's shared-memory
// writes, then wait for all CTAs (acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The float at the same shared-memory offset as `local`, in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_cluster_f32(const float* local, unsigned rank) {
  unsigned remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

template <typename Op>
__global__ void __launch_bounds__(kClusterThreads) k_reduce_cluster(ContigParams p) {
  pdl_begin();
  constexpr int U = kClusterLoads;
  constexpr int64_t S = kClusterThreads;
  __shared__ float sh[kClusterThreads / 32];
  __shared__ float s_part;
  const int t = threadIdx.x;
  const unsigned rank = cluster_ctarank();  // the grid is one cluster
  const int64_t start = (int64_t)rank * p.chunk_len;
  const int64_t len = max((int64_t)0, min(p.chunk_len, p.seg_len - start));
  const float* a = p.x + start;
  // Peel up to three leading floats so the body is 16-byte aligned.
  int64_t head = (int64_t)((0u - (unsigned)(uintptr_t)a) & 15u) >> 2;
  if (head > len) head = len;
  const int64_t nvec = (len - head) >> 2;  // at most U * S
  const int tail = (int)((len - head) & 3);
  const float* av = a + head;
  float4 r[U];
#pragma unroll
  for (int u = 0; u < U; ++u)
    if (t + u * S < nvec) r[u] = ld_stream4(av + 4 * (t + u * S));
  float sv[U];
#pragma unroll
  for (int u = 0; u < U; ++u) sv[u] = t + u * S < nvec ? reduce4<Op>(r[u]) : Op::identity();
  float v = tree_reduce<Op, U>(sv);
  if (t < head) v = Op::combine(v, Op::prep(ld_plain(a + t)));
  if (t < tail) v = Op::combine(v, Op::prep(ld_plain(av + 4 * nvec + t)));
  v = block_reduce<Op, kClusterThreads>(v, sh);
  if (t == 0) s_part = v;
  cluster_sync();
  if (rank == 0 && t < 32) {
    float q = t < p.chunks ? ld_cluster_f32(&s_part, (unsigned)t) : Op::identity();
    q = warp_reduce<Op>(q);  // the CTAs' results in a fixed tree
    if (t == 0) st_plain(p.out, finish(q, p.epi, p.seg_len));
  }
  cluster_sync();  // every CTA's shared memory stays alive until CTA 0 has read it
}

// ---------------------------------------------------------------------------
// Short rows: one warp per row, rows strided over the grid.
// ---------------------------------------------------------------------------
template <typename Op>
__global__ void __launch_bounds__(kThreads) k_reduce_rows_warp(RowsWarpParams p) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int64_t first = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  for (int64_t row = first; row < p.rows; row += nwarps) {
    const float* a = p.x + row * p.len;
    BlockedAcc<kFold, Op> acc;
    int64_t j = lane;
    for (; j + 7 * 32 < p.len; j += 8 * 32) {
      float r[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) r[u] = Op::prep(ld_stream1(a + j + u * 32));
      acc.add(tree_reduce<Op, 8>(r));
    }
    for (; j < p.len; j += 32) acc.add(Op::prep(ld_stream1(a + j)));
    const float v = warp_reduce<Op>(acc.total());
    if (lane == 0) st_plain(p.out + row, finish(v, p.epi, p.len));
  }
}

// ---------------------------------------------------------------------------
// Axis sum, inner > 1: warps across columns, loop over the reduce dim.
// ---------------------------------------------------------------------------
template <int VEC, int WY>
struct ColsShape {
  static constexpr int WX = 8 / WY;            // warps across columns
  static constexpr int CW = WX * 32 * VEC;     // columns per block
};

template <int VEC, int WY, int U, typename Op>
__global__ void __launch_bounds__(kThreads) k_reduce_cols(ColsParams p) {
  pdl_begin();
  using Sh = ColsShape<VEC, WY>;
  constexpr int WX = Sh::WX;
  constexpr int CW = Sh::CW;
  __shared__ __align__(16) float sh[1024];
  __shared__ int am_last;

  int64_t b = blockIdx.x;
  const int64_t ct = b % p.col_tiles;
  b /= p.col_tiles;
  const int64_t s = b % p.splits;
  const int64_t o = b / p.splits;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wx = warp % WX;
  const int wy = warp / WX;
  const int jloc = wx * 32 * VEC + lane * VEC;
  const int64_t col = ct * CW + jloc;
  const int64_t r0 = s * p.rows_per_split;
  const int64_t r1 = min(r0 + p.rows_per_split, p.reduce);
  const int64_t inner = p.inner;

  float res[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) res[c] = Op::identity();

  if (col < inner) {
    const float* xc = p.x + o * p.reduce * inner + col;
    BlockedAcc<kFold, Op> acc[VEC];
    int64_t r = r0 + wy;
    for (; r + (U - 1) * WY < r1; r += U * WY) {
      if constexpr (VEC == 4) {
        float4 q[U];
#pragma unroll
        for (int u = 0; u < U; ++u) q[u] = ld_stream4(xc + (r + u * WY) * inner);
        float e[4][U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          e[0][u] = Op::prep(q[u].x);
          e[1][u] = Op::prep(q[u].y);
          e[2][u] = Op::prep(q[u].z);
          e[3][u] = Op::prep(q[u].w);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c].add(tree_reduce<Op, U>(e[c]));
      } else {
        float q[U];
#pragma unroll
        for (int u = 0; u < U; ++u) q[u] = Op::prep(ld_stream1(xc + (r + u * WY) * inner));
        acc[0].add(tree_reduce<Op, U>(q));
      }
    }
    for (; r < r1; r += WY) {
      if constexpr (VEC == 4) {
        const float4 q = ld_stream4(xc + r * inner);
        acc[0].add(Op::prep(q.x));
        acc[1].add(Op::prep(q.y));
        acc[2].add(Op::prep(q.z));
        acc[3].add(Op::prep(q.w));
      } else {
        acc[0].add(Op::prep(ld_stream1(xc + r * inner)));
      }
    }
#pragma unroll
    for (int c = 0; c < VEC; ++c) res[c] = acc[c].total();
  }

  // Combine the WY row groups of the block in a fixed tree.
  if constexpr (WY > 1) {
#pragma unroll
    for (int c = 0; c < VEC; ++c) sh[wy * CW + jloc + c] = res[c];
    __syncthreads();
    if (wy == 0) {
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        float v[WY];
#pragma unroll
        for (int k = 0; k < WY; ++k) v[k] = sh[k * CW + jloc + c];
        res[c] = tree_reduce<Op, WY>(v);
      }
    }
  }

  if (p.splits == 1) {
    if (wy == 0) {
      float* outp = p.out + o * inner;
#pragma unroll
      for (int c = 0; c < VEC; ++c)
        if (col + c < inner) st_plain(outp + col + c, finish(res[c], p.epi, p.reduce));
    }
    return;
  }

  // Split reduce: publish this slice's column sums, then let the last block of
  // (o, ct) add the slices in slice order.
  float* part_base = p.partials + (o * p.splits) * (int64_t)p.col_tiles * CW + ct * CW;
  const int64_t slice_stride = (int64_t)p.col_tiles * CW;
  if (wy == 0) {
    float* mine = part_base + s * slice_stride;
#pragma unroll
    for (int c = 0; c < VEC; ++c) st_plain(mine + jloc + c, res[c]);
    if (p.keep_partials) return;  // the slice sums are the result
    __threadfence();
  }
  if (p.keep_partials) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = take_count(p.tickets + o * p.col_tiles + ct);
    am_last = (prev == (unsigned)(p.splits - 1));
  }
  __syncthreads();
  if (!am_last) return;
  __threadfence();

  constexpr int Q = CW / 4;            // float4 columns of the tile
  constexpr int G = kThreads / Q;      // slice groups
  const int q = threadIdx.x % Q;
  const int g = threadIdx.x / Q;
  BlockedAcc<kFold, Op> acc4[4];
  {
    int64_t k = g;
    const int64_t S = p.splits;
    for (; k + 3 * G < S; k += 4 * G) {
      float4 r[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) r[u] = ld_cg4(part_base + (k + u * G) * slice_stride + 4 * q);
      float e[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        e[0][u] = r[u].x;
        e[1][u] = r[u].y;
        e[2][u] = r[u].z;
        e[3][u] = r[u].w;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) acc4[c].add(tree_reduce<Op, 4>(e[c]));
    }
    for (; k < S; k += G) {
      const float4 r = ld_cg4(part_base + k * slice_stride + 4 * q);
      acc4[0].add(r.x);
      acc4[1].add(r.y);
      acc4[2].add(r.z);
      acc4[3].add(r.w);
    }
  }
  __syncthreads();  // sh may still be read by the row-group combine above
#pragma unroll
  for (int c = 0; c < 4; ++c) sh[g * CW + 4 * q + c] = acc4[c].total();
  __syncthreads();
  if (threadIdx.x < Q) {
    float* outp = p.out + o * inner;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v[G];
#pragma unroll
      for (int k = 0; k < G; ++k) v[k] = sh[k * CW + 4 * q + c];
      const float tot = tree_reduce<Op, G>(v);
      const int64_t cc = ct * CW + 4 * q + c;
      if (cc < inner) st_plain(outp + cc, finish(tot, p.epi, p.reduce));
    }
    if (threadIdx.x == 0) st_plain(p.tickets + o * p.col_tiles + ct, 0u);
  }
}

// Unroll depth (rows or vectors in flight per thread) of each variant.
constexpr int kColsU = 8;

__global__ void k_fill(float* out, int64_t n, float value) {
  pdl_begin();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    st_plain(out + i, value);
}

template <typename K>
int occupancy_of(K kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess) return 0;
  return n;
}

template <typename Op>
cudaError_t contig_op(int variant, const ContigParams& p, dim3 g, cudaStream_t s) {
  if constexpr (std::is_same<Op, OpSum>::value) {
    switch (variant) {
      case kContigU4: launch_pdl(k_reduce_contig<4, Op>, g, kThreads, 0, s, p); return cudaGetLastError();
      case kContigU8: launch_pdl(k_reduce_contig<8, Op>, g, kThreads, 0, s, p); return cudaGetLastError();
      default: break;
    }
  }
  if (variant != kContigU16) return cudaErrorInvalidValue;
  launch_pdl(k_reduce_contig<16, Op>, g, kThreads, 0, s, p);
  return cudaGetLastError();
}

template <typename Op>
cudaError_t cols_op(int variant, const ColsParams& p, dim3 g, cudaStream_t s) {
  if constexpr (std::is_same<Op, OpSum>::value) {
    switch (variant) {
      case kColsV1W1: launch_pdl(k_reduce_cols<1, 1, kColsU, Op>, g, kThreads, 0, s, p); return cudaGetLastError();
      case kColsV1W8: launch_pdl(k_reduce_cols<1, 8, kColsU, Op>, g, kThreads, 0, s, p); return cudaGetLastError();
      case kColsV4W1: launch_pdl(k_reduce_cols<4, 1, kColsU, Op>, g, kThreads, 0, s, p); return cudaGetLastError();
      case kColsV4W8: launch_pdl(k_reduce_cols<4, 8, kColsU, Op>, g, kThreads, 0, s, p); return cudaGetLastError();
      default: break;
    }
  }
  switch (variant) {
    case kColsV1W4: launch_pdl(k_reduce_cols<1, 4, kColsU, Op>, g, kThreads, 0, s, p); break;
    case kColsV4W4: launch_pdl(k_reduce_cols<4, 4, kColsU, Op>, g, kThreads, 0, s, p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

int cols_block_width(int variant) {
  switch (variant) {
    case kColsV1W1: return ColsShape<1, 1>::CW;
    case kColsV1W4: return ColsShape<1, 4>::CW;
    case kColsV1W8: return ColsShape<1, 8>::CW;
    case kColsV4W1: return ColsShape<4, 1>::CW;
    case kColsV4W4: return ColsShape<4, 4>::CW;
    case kColsV4W8: return ColsShape<4, 8>::CW;
    default: return 0;
  }
}

cudaError_t launch_reduce_contig(int variant, int op, const ContigParams& p, int64_t grid,
                                 cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (op) {
    case kOpSum: return contig_op<OpSum>(variant, p, g, s);
    case kOpSumSq: return contig_op<OpSumSq>(variant, p, g, s);
    case kOpMax: return contig_op<OpMax>(variant, p, g, s);
    case kOpMin: return contig_op<OpMin>(variant, p, g, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename Op>
cudaError_t cluster_op(const ContigParams& p, int ctas, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kClusterThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_begin
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_reduce_cluster<Op>, p);
}

cudaError_t launch_reduce_cluster(int op, const ContigParams& p, int ctas, cudaStream_t s) {
  if (ctas < 1 || ctas > kClusterMaxCtas || p.chunks != ctas ||
      p.chunk_len > (int64_t)kClusterThreads * kClusterLoads * 4)
    return cudaErrorInvalidValue;
  switch (op) {
    case kOpSum: return cluster_op<OpSum>(p, ctas, s);
    case kOpSumSq: return cluster_op<OpSumSq>(p, ctas, s);
    case kOpMax: return cluster_op<OpMax>(p, ctas, s);
    case kOpMin: return cluster_op<OpMin>(p, ctas, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_reduce_rows_warp(int op, const RowsWarpParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (op) {
    case kOpSum: launch_pdl(k_reduce_rows_warp<OpSum>, g, kThreads, 0, s, p); break;
    case kOpSumSq: launch_pdl(k_reduce_rows_warp<OpSumSq>, g, kThreads, 0, s, p); break;
    case kOpMax: launch_pdl(k_reduce_rows_warp<OpMax>, g, kThreads, 0, s, p); break;
    case kOpMin: launch_pdl(k_reduce_rows_warp<OpMin>, g, kThreads, 0, s, p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_reduce_cols(int variant, int op, const ColsParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (op) {
    case kOpSum: return cols_op<OpSum>(variant, p, g, s);
    case kOpSumSq: return cols_op<OpSumSq>(variant, p, g, s);
    case kOpMax: return cols_op<OpMax>(variant, p, g, s);
    case kOpMin: return cols_op<OpMin>(variant, p, g, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fill(float* out, int64_t n, float value, cudaStream_t s) {
  const int64_t blocks = std::min<int64_t>((n + kThreads - 1) / kThreads, 4096);
  launch_pdl(k_fill, dim3((unsigned)std::max<int64_t>(1, blocks)), kThreads, 0, s, out, n, value);
  return cudaGetLastError();
}

namespace {

template <typename Op>
int occ_contig(int variant) {
  if constexpr (std::is_same<Op, OpSum>::value) {
    if (variant == kContigU4) return occupancy_of(k_reduce_contig<4, Op>);
    if (variant == kContigU8) return occupancy_of(k_reduce_contig<8, Op>);
  }
  return variant == kContigU16 ? occupancy_of(k_reduce_contig<16, Op>) : 0;
}

template <typename Op>
int occ_cols(int variant) {
  if constexpr (std::is_same<Op, OpSum>::value) {
    switch (variant) {
      case kColsV1W1: return occupancy_of(k_reduce_cols<1, 1, kColsU, Op>);
      case kColsV1W8: return occupancy_of(k_reduce_cols<1, 8, kColsU, Op>);
      case kColsV4W1: return occupancy_of(k_reduce_cols<4, 1, kColsU, Op>);
      case kColsV4W8: return occupancy_of(k_reduce_cols<4, 8, kColsU, Op>);
      default: break;
    }
  }
  if (variant == kColsV1W4) return occupancy_of(k_reduce_cols<1, 4, kColsU, Op>);
  if (variant == kColsV4W4) return occupancy_of(k_reduce_cols<4, 4, kColsU, Op>);
  return 0;
}

}  // namespace

int occupancy_reduce_contig(int variant, int op) {
  switch (op) {
    case kOpSum: return occ_contig<OpSum>(variant);
    case kOpSumSq: return occ_contig<OpSumSq>(variant);
    case kOpMax: return occ_contig<OpMax>(variant);
    case kOpMin: return occ_contig<OpMin>(variant);
    default: return 0;
  }
}

int occupancy_reduce_rows_warp(int op) {
  switch (op) {
    case kOpSum: return occupancy_of(k_reduce_rows_warp<OpSum>);
    case kOpSumSq: return occupancy_of(k_reduce_rows_warp<OpSumSq>);
    case kOpMax: return occupancy_of(k_reduce_rows_warp<OpMax>);
    case kOpMin: return occupancy_of(k_reduce_rows_warp<OpMin>);
    default: return 0;
  }
}

int occupancy_reduce_cols(int variant, int op) {
  switch (op) {
    case kOpSum: return occ_cols<OpSum>(variant);
    case kOpSumSq: return occ_cols<OpSumSq>(variant);
    case kOpMax: return occ_cols<OpMax>(variant);
    case kOpMin: return occ_cols<OpMin>(variant);
    default: return 0;
  }
}

}  // namespace lr
