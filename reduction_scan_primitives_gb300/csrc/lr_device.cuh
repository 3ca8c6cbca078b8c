// lr_device.cuh -- device helpers shared by the libreduce kernels (sm_103a).
//
// Warp-level trees use __shfl_down_sync, as in "Seven-step reduction: 30x from
// one kernel" (V7, two-level warp-shuffle reduction) and the warp-shuffle
// design decision of the "High-Performance Reduction Kernels" README.  Loads
// of the input stream are 128-bit and bypass L1 allocation; outputs of the
// scan are written with an evict-first hint.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace lr {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// Global memory access (hand-written PTX).
// ---------------------------------------------------------------------------

// 128-bit load of read-only data through the non-coherent path, without
// allocating in L1 (the stream is touched once).  p must be 16-byte aligned.
__device__ __forceinline__ float4 ld_stream4(const float* p) {
  float4 v;
  asm("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "l"(p));
  return v;
}

// 32-bit load of read-only data, no L1 allocation.
__device__ __forceinline__ float ld_stream1(const float* p) {
  float v;
  asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// 128-bit store with the evict-first (streaming) hint.  p must be 16-byte aligned.
__device__ __forceinline__ void st_stream4(float* p, float4 v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_stream1(float* p, float v) {
  asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Load from L2 (bypassing L1), used for partial sums written by other blocks
// of the same launch.
__device__ __forceinline__ float ld_cg1(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float4 ld_cg4(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}

// ---------------------------------------------------------------------------
// Inter-block signalling (GPU scope).  Used by the look-back scan, whose
// blocks publish values that other blocks of the same launch wait for.
// ---------------------------------------------------------------------------

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// A 64-bit word that carries its own validity (an epoch next to the value)
// needs no ordering with other data, so relaxed single-copy-atomic accesses
// suffice and no fence is paid on either side.
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// Bulk copies (TMA engine, 1D) into shared memory, completed on an mbarrier.
// ---------------------------------------------------------------------------

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier shared-memory accesses before later bulk copies.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// One non-blocking probe of phase `parity` of the barrier.
__device__ __forceinline__ bool mbar_try_wait_parity(unsigned long long* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// to shared memory; completion is signalled as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src_gmem, unsigned bytes,
                                          unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// Summation building blocks.  Every tree below has a fixed shape, so a given
// input always produces the same bits.
// ---------------------------------------------------------------------------

__device__ __forceinline__ float sum4(float4 v) { return (v.x + v.y) + (v.z + v.w); }

// Pairwise sum of a small register array, fixed shape.
template <int N>
__device__ __forceinline__ float tree_sum(const float* v) {
  if constexpr (N == 1) {
    return v[0];
  } else {
    constexpr int H = N / 2;
    return tree_sum<H>(v) + tree_sum<N - H>(v + H);
  }
}

// Warp sum: lane 0 receives the sum of v over the 32 lanes.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(kFullMask, v, o);
  return v;
}

// Block sum for NT threads (NT a multiple of 32, at most 1024).  `sh` holds
// NT/32 floats.  The result is valid in thread 0.  The caller must place a
// __syncthreads() between two uses of the same `sh`.
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* sh) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if constexpr (NW == 1) {
    return v;
  } else {
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    float r = 0.f;
    if (warp == 0) {
      r = lane < NW ? sh[lane] : 0.f;
#pragma unroll
      for (int o = NW / 2; o > 0; o >>= 1) r += __shfl_down_sync(kFullMask, r, o);
    }
    return r;
  }
}

// Three-level accumulator.  A plain running fp32 sum over m terms has an
// addition chain of length m, and its worst-case rounding error grows with m.
// Folding the running sum into a second, then a third register every K terms
// keeps every chain at most K + K + m/K^2 long, at the cost of two extra adds
// per K terms.  The fold points depend only on the number of terms, so the
// result is deterministic.
template <int K>
struct BlockedAcc {
  float lo = 0.f, mid = 0.f, hi = 0.f;
  int n_lo = 0, n_mid = 0;
  __device__ __forceinline__ void add(float v) {
    lo += v;
    if (++n_lo == K) {
      mid += lo;
      lo = 0.f;
      n_lo = 0;
      if (++n_mid == K) {
        hi += mid;
        mid = 0.f;
        n_mid = 0;
      }
    }
  }
  __device__ __forceinline__ float total() const { return hi + (mid + lo); }
};

}  // namespace lr
