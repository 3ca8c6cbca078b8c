// lr_contig.cuh -- the contiguous-chunk reduction kernel (1D and long rows),
// shared by the translation units that launch it.  Each including file gets
// its own instantiation (internal linkage).
//
// Design, by source: "High-Performance Reduction Kernels" README ('Key design
// decisions': float4 loads, warp-shuffle trees, one float per warp in shared
// memory, contiguous block assignment; 'Optimization: ILP4 accumulator':
// several independent loads in flight per thread) and "Seven-step reduction:
// 30x from one kernel" (V7), with the atomicAdd finish replaced by a
// deterministic last-block combine.
#pragma once

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

constexpr int kFold = 16;  // blocked-accumulator fold length

// Reduce p[start], p[start + stride], ... (< n), eight loads in flight, fixed
// order.  The data was written by other blocks of this launch, so it is read
// from L2.  The values are partial results, already prepped.
template <typename Op>
__device__ __forceinline__ float reduce_strided_cg(const float* p, int64_t n, int64_t start,
                                                   int64_t stride) {
  BlockedAcc<kFold, Op> acc;
  int64_t k = start;
  for (; k + 7 * stride < n; k += 8 * stride) {
    float r[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) r[u] = ld_cg1(p + k + u * stride);
    acc.add(tree_reduce<Op, 8>(r));
  }
  for (; k < n; k += stride) acc.add(ld_cg1(p + k));
  return acc.total();
}

// ---------------------------------------------------------------------------
// 1D reduction / long rows: one block per (segment, chunk).
// ---------------------------------------------------------------------------
template <int U, typename Op>
__global__ void __launch_bounds__(kThreads) k_reduce_contig(ContigParams p) {
  pdl_begin();
  __shared__ float sh[kThreads / 32];
  __shared__ int am_last;
  const int t = threadIdx.x;
  const int64_t unit = blockIdx.x;
  const int64_t seg = unit / p.chunks;
  const int64_t c = unit - seg * p.chunks;
  const float* a = p.x + seg * p.seg_len + c * p.chunk_len;
  const int64_t len = min(p.chunk_len, p.seg_len - c * p.chunk_len);

  // Peel up to three leading floats so the body is 16-byte aligned.
  int64_t head = (int64_t)((0u - (unsigned)(uintptr_t)a) & 15u) >> 2;
  if (head > len) head = len;
  const int64_t nvec = (len - head) >> 2;
  const int tail = (int)((len - head) & 3);
  const float* av = a + head;

  BlockedAcc<kFold, Op> acc;
  constexpr int64_t S = kThreads;
  int64_t i = t;
  for (; i + (U - 1) * S < nvec; i += U * S) {
    float4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) r[u] = ld_stream4(av + 4 * (i + u * S));
    float s[U];
#pragma unroll
    for (int u = 0; u < U; ++u) s[u] = reduce4<Op>(r[u]);
    acc.add(tree_reduce<Op, U>(s));
  }
  if (i < nvec) {
    // The remainder (fewer than U loads per thread) is issued all at once, so
    // a short chunk costs one memory round trip rather than one per load.
    // (Measured against batches of 6 and 8, which need fewer registers: the
    // same within 10% from 1e4 to 1e9 elements, ahead at 1e6.)
    float4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i + u * S < nvec) r[u] = ld_stream4(av + 4 * (i + u * S));
    float s[U];
#pragma unroll
    for (int u = 0; u < U; ++u) s[u] = i + u * S < nvec ? reduce4<Op>(r[u]) : Op::identity();
    acc.add(tree_reduce<Op, U>(s));
  }
  float v = acc.total();
  if (t < head) v = Op::combine(v, Op::prep(ld_plain(a + t)));
  if (t < tail) v = Op::combine(v, Op::prep(ld_plain(av + 4 * nvec + t)));

  v = block_reduce<Op, kThreads>(v, sh);
  if (p.chunks == 1) {
    if (t == 0) st_plain(p.out + seg, finish(v, p.epi, p.seg_len));
    return;
  }
  if (t == 0) {
    st_plain(p.partials + unit, v);
    __threadfence();
    const unsigned prev = take_count(p.tickets + seg);
    am_last = (prev == (unsigned)(p.chunks - 1));
  }
  __syncthreads();
  if (!am_last) return;
  __threadfence();
  float s = reduce_strided_cg<Op>(p.partials + seg * p.chunks, p.chunks, t, kThreads);
  s = block_reduce<Op, kThreads>(s, sh);
  if (t == 0) {
    st_plain(p.out + seg, finish(s, p.epi, p.seg_len));
    st_plain(p.tickets + seg, 0u);  // ready for the next launch
  }
}

}  // namespace
}  // namespace lr
