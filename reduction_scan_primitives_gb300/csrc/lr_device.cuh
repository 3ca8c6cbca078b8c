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

#include "lr_internal.h"

namespace lr {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// Debug builds (LR_DEBUG, the library's separate debug build): every global
// access made through the helpers below, and the shared-memory slots of the
// short-row kernels, is checked before it happens.  The host registers the
// byte ranges [lo, hi) of each call's buffers (inputs, outputs, scratch);
// an access outside all of them, a shared-memory index outside its buffer,
// or a misaligned vector access is recorded (flag bits and the first
// offending address) and skipped -- a load reads zeros -- never trapped.
// libreduce_check() reports it.  Release builds compile none of this.
// ---------------------------------------------------------------------------
#ifdef LR_DEBUG
extern __device__ LrDebug g_lr_debug;

__device__ __forceinline__ void dbg_record(unsigned bit, unsigned long long addr) {
  atomicOr(&g_lr_debug.flags, bit);
  atomicCAS(&g_lr_debug.first_bad, 0ull, addr | 1ull);  // | 1: a recorded zero address stays visible
}
// True when [p, p + bytes) lies inside one registered range (and p is aligned
// to `align` bytes); else records the access.  A load may cover the rest of
// the 16-byte granules at a range's two ends: the float4 kernels read a row
// edge's whole granule by design (it lies in the same page as the element it
// holds) and mask the elements outside; a store must stay inside the range.
__device__ __forceinline__ bool dbg_global(const void* p, unsigned bytes, unsigned align, bool load) {
  const unsigned long long a = reinterpret_cast<unsigned long long>(p);
  if (a & (align - 1)) {
    dbg_record(kDbgMisaligned, a);
    return false;
  }
#pragma unroll
  for (int i = 0; i < kDbgRanges; ++i) {
    const unsigned long long lo = load ? g_lr_debug.lo[i] & ~15ull : g_lr_debug.lo[i];
    const unsigned long long hi = load ? (g_lr_debug.hi[i] + 15) & ~15ull : g_lr_debug.hi[i];
    if (g_lr_debug.hi[i] > g_lr_debug.lo[i] && a >= lo && a + bytes <= hi) return true;
  }
  dbg_record(kDbgGlobal, a);
  return false;
}
// True when element index i (width w elements) lies inside a shared buffer of n elements.
__device__ __forceinline__ bool dbg_shared(long long i, int w, long long n, const void* p) {
  if (i >= 0 && i + w <= n) return true;
  dbg_record(kDbgShared, reinterpret_cast<unsigned long long>(p));
  return false;
}
#define LR_DBG_GLOBAL(p, bytes, align) ::lr::dbg_global((p), (bytes), (align), true)
#define LR_DBG_GLOBAL_ST(p, bytes, align) ::lr::dbg_global((p), (bytes), (align), false)
#define LR_DBG_SHARED(i, w, n, p) ::lr::dbg_shared((i), (w), (n), (p))
#else
#define LR_DBG_GLOBAL(p, bytes, align) true
#define LR_DBG_GLOBAL_ST(p, bytes, align) true
#define LR_DBG_SHARED(i, w, n, p) true
#endif

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel is launched so that it may
// start while the previous kernel in its stream is still finishing; its first
// statement waits until that kernel has completed and its memory operations
// are visible (a no-op after a plain launch), so no access of this kernel
// overlaps the previous one.  It then lets the next kernel of the stream
// begin its launch, which completes once every block of this grid has begun.
// What overlaps is launch processing and block start-up, nothing else.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Global memory access (hand-written PTX).
// ---------------------------------------------------------------------------

// 128-bit load of read-only data through the non-coherent path, without
// allocating in L1 (the stream is touched once).  p must be 16-byte aligned.
__device__ __forceinline__ float4 ld_stream4(const float* p) {
  float4 v;
  if (!LR_DBG_GLOBAL(p, 16, 16)) return make_float4(0.f, 0.f, 0.f, 0.f);
  asm("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "l"(p));
  return v;
}

// 32-bit load of read-only data, no L1 allocation.
__device__ __forceinline__ float ld_stream1(const float* p) {
  float v;
  if (!LR_DBG_GLOBAL(p, 4, 4)) return 0.f;
  asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// 128-bit store with the evict-first (streaming) hint.  p must be 16-byte aligned.
__device__ __forceinline__ void st_stream4(float* p, float4 v) {
  if (!LR_DBG_GLOBAL_ST(p, 16, 16)) return;
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_stream1(float* p, float v) {
  if (!LR_DBG_GLOBAL_ST(p, 4, 4)) return;
  asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Load from L2 (bypassing L1), used for partial sums written by other blocks
// of the same launch.
__device__ __forceinline__ float ld_cg1(const float* p) {
  if (!LR_DBG_GLOBAL(p, 4, 4)) return 0.f;
  return __ldcg(p);
}
__device__ __forceinline__ float4 ld_cg4(const float* p) {
  if (!LR_DBG_GLOBAL(p, 16, 16)) return make_float4(0.f, 0.f, 0.f, 0.f);
  return __ldcg(reinterpret_cast<const float4*>(p));
}

// Plain global accesses of the kernels (outputs, partials, carries, edge
// elements), checked in debug builds like the helpers above.
template <typename T>
__device__ __forceinline__ T ld_plain(const T* p) {
  if (!LR_DBG_GLOBAL(p, sizeof(T), sizeof(T))) return T(0);
  return *p;
}
template <typename T>
__device__ __forceinline__ void st_plain(T* p, T v) {
  if (!LR_DBG_GLOBAL_ST(p, sizeof(T), sizeof(T))) return;
  *p = v;
}

// ---------------------------------------------------------------------------
// Inter-block signalling (GPU scope).  Used by the look-back scan, whose
// blocks publish values that other blocks of the same launch wait for.
// ---------------------------------------------------------------------------

// A 64-bit word that carries its own validity (an epoch next to the value)
// needs no ordering with other data, so relaxed single-copy-atomic accesses
// suffice and no fence is paid on either side.
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  if (!LR_DBG_GLOBAL(p, 8, 8)) return 0ull;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  if (!LR_DBG_GLOBAL_ST(p, 8, 8)) return;
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  if (!LR_DBG_GLOBAL(p, 4, 4)) return 0u;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Look-back node words: {epoch:32, fp32 bits:32}.  A word counts only if its
// epoch is the current launch's, so node buffers never need clearing.
__device__ __forceinline__ unsigned long long pack_node(unsigned epoch, float v) {
  return ((unsigned long long)epoch << 32) | (unsigned long long)__float_as_uint(v);
}

// Poll a node until it carries this launch's epoch (or give up).
__device__ __forceinline__ float wait_node(const unsigned long long* node, unsigned epoch,
                                           int64_t limit, const unsigned* abort_word, bool* fail) {
  unsigned ns = 0;
  for (int64_t it = 0;; ++it) {
    const unsigned long long word = ld_relaxed_u64(node);
    if ((unsigned)(word >> 32) == epoch) return __uint_as_float((unsigned)word);
    if (it >= limit || ld_relaxed_u32(abort_word) == epoch) {
      *fail = true;
      return 0.f;
    }
    if (it >= 64) {  // spin first, then back off gently
      ns = ns ? (ns < 256 ? 2 * ns : ns) : 32;
      __nanosleep(ns);
    }
  }
}

// The P class words of one look-back node (consecutive words from `node`):
// all P loads are issued at once, then only the words not yet carrying this
// launch's epoch are polled (bounded, as wait_node).
// In two steps, so that other work hides the loads' latency: load_node_classes
// issues the loads, settle_node_classes polls the words that did not carry
// the epoch yet.
template <int P>
__device__ __forceinline__ void load_node_classes(const unsigned long long* node, unsigned long long (&word)[P]) {
#pragma unroll
  for (int c = 0; c < P; ++c) word[c] = ld_relaxed_u64(node + c);
}
template <int P>
__device__ __forceinline__ void settle_node_classes(const unsigned long long* node, const unsigned long long (&word)[P],
                                                    unsigned epoch, int64_t limit, const unsigned* abort_word,
                                                    bool* fail, float (&out)[P]) {
#pragma unroll
  for (int c = 0; c < P; ++c)
    out[c] = (unsigned)(word[c] >> 32) == epoch ? __uint_as_float((unsigned)word[c])
                                                : wait_node(node + c, epoch, limit, abort_word, fail);
}
template <int P>
__device__ __forceinline__ void wait_node_classes(const unsigned long long* node, unsigned epoch, int64_t limit,
                                                  const unsigned* abort_word, bool* fail, float (&out)[P]) {
  unsigned long long word[P];
  load_node_classes<P>(node, word);
  settle_node_classes<P>(node, word, epoch, limit, abort_word, fail, out);
}

// a[i] selected by a run-time index (registers cannot be indexed at run time).
template <int P>
__device__ __forceinline__ float pick_class(const float (&a)[P], int i) {
  float r = a[0];
#pragma unroll
  for (int c = 1; c < P; ++c)
    if (i == c) r = a[c];
  return r;
}

// Fixed pairwise tree over the 32 lanes (adjacent pairs first); lane 0 gets it.
__device__ __forceinline__ float warp_tree_adjacent(float v) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) v += __shfl_down_sync(kFullMask, v, o);
  return v;
}

// An integer ticket: atomicAdd(p, 1) (debug builds: a ticket outside the
// call's scratch is recorded and reads as ~0u, the caller then takes no part
// in the combine).
__device__ __forceinline__ unsigned take_count(unsigned* p) {
  if (!LR_DBG_GLOBAL_ST(p, 4, 4)) return ~0u;
  return atomicAdd(p, 1u);
}

// Tickets and the launch's epoch (the tag that tells this launch's node words
// from older ones) share one 64-bit device word: epoch in the high half, the
// ticket counter in the low half.  One atomicAdd gives a block both; the
// block with the last ticket -- every other block has taken its ticket --
// resets the counter and advances the epoch (0 is reserved for "never
// written").  Kept on the device rather than passed by the host, so a launch
// captured in a CUDA graph gets a new epoch at every replay.
struct Ticket {
  unsigned ticket, epoch;
};
__device__ __forceinline__ Ticket take_ticket(unsigned long long* word) {
  // Debug builds: a ticket word outside the call's scratch gives a ticket past
  // every launch's range (and below 2^31, so no kernel mistakes it for a
  // tile of its own), and the block leaves without starting a copy.
  if (!LR_DBG_GLOBAL_ST(word, 8, 8)) return Ticket{0x7fffffffu, 1u};
  const unsigned long long old = atomicAdd(word, 1ull);
  const unsigned e = (unsigned)(old >> 32);
  return Ticket{(unsigned)old, e == 0 ? 1u : e};
}
__device__ __forceinline__ void next_launch(unsigned long long* word, unsigned epoch) {
  atomicExch(word, (unsigned long long)(epoch + 1 == 0 ? 1u : epoch + 1) << 32);
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

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// A plain arrival (no transaction bytes): completes the current phase of a
// barrier initialised with count 1 when no copy is started for it.
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for this block's own bulk or tensor copy (from this GPU's memory) to
// complete phase `parity` of `bar`.  Such a copy lands within microseconds
// and depends on no other block, so this wait is bounded by time -- two
// seconds of the global timer, far beyond any copy -- and not by the
// adjustable poll limit of the flag waits: a short poll limit (as the timeout
// tests set) must never let a block leave while its copy still writes into
// its shared memory.  Returns false only if the copy never completed.
constexpr unsigned long long kCopyWaitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait_copy(unsigned long long* bar, unsigned parity) {
  if (mbar_try_wait_parity(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait_parity(bar, parity))
    if (global_ns() - t0 > kCopyWaitNs) return false;
  return true;
}

// Orders this thread's earlier shared-memory accesses (generic proxy) before
// bulk copies issued after the next block barrier (async proxy): a buffer
// that threads have read or written is refilled by the TMA engine only after
// every thread has fenced and the block has synchronised.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// to shared memory; completion is signalled as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src_gmem, unsigned bytes,
                                          unsigned long long* bar) {
#ifdef LR_DEBUG
  // A source range outside the call's buffers: no copy; the expected bytes
  // are completed on the barrier by hand, so its waiters still finish.
  if (!LR_DBG_GLOBAL(src_gmem, bytes, 16)) {
    asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
    return;
  }
#endif
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from shared
// to global memory as one bulk copy of the issuing thread's current bulk
// group.  The shared source may be written again only after
// bulk_store_wait_read; the issuing thread waits with bulk_store_wait_all
// before its block leaves.  Writers of the source fence with
// fence_proxy_async_smem and synchronise with the issuer first.
__device__ __forceinline__ void bulk_store(void* dst_gmem, const void* src_smem, unsigned bytes) {
  if (!LR_DBG_GLOBAL_ST(dst_gmem, bytes, 16)) return;  // debug: a destination outside the call's buffers
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
               "r"(smem_u32(src_smem)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's bulk stores have read their shared sources.
__device__ __forceinline__ void bulk_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's bulk stores are complete.
__device__ __forceinline__ void bulk_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Tiled tensor copy (TMA engine) of one 3-D box into shared memory, completed
// on an mbarrier.  `tmap` is the generic address of a tensor map held in
// kernel parameter space (__grid_constant__); c0 is the innermost coordinate
// (c0 * element size must be a multiple of 16 bytes), c1 and c2 may lie
// outside the tensor, whose elements there arrive as zeros.
__device__ __forceinline__ void tma_load_3d(void* dst_smem, const void* tmap, int c0, int c1, int c2,
                                            unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst_smem)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Per-thread asynchronous copies into shared memory (cp.async).  The first
// `src_bytes` of the copy come from global memory and the rest is filled with
// zeros, so src_bytes == 0 writes a zero item without reading anything (`src`
// must still be a valid address).  Completion: commit_group, then wait_group.
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src, unsigned src_bytes) {
  if (src_bytes && !LR_DBG_GLOBAL(src, 16, 16)) src_bytes = 0;  // debug: a bad source fills zeros
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst_smem)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst_smem, const void* src, unsigned src_bytes) {
  if (src_bytes && !LR_DBG_GLOBAL(src, 4, 4)) src_bytes = 0;  // debug: a bad source fills zeros
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst_smem)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// Reduction operators.  `prep` maps a loaded element to the value that is
// combined (x*x for a sum of squares); `combine` is associative up to
// rounding; `identity` is the value of an empty reduction.  Max and min
// propagate NaN (a NaN operand wins), like the comparison-based reductions
// of most array libraries; on ties they keep one operand, chosen by position.
// ---------------------------------------------------------------------------
struct OpSum {
  static __device__ __forceinline__ float identity() { return 0.f; }
  static __device__ __forceinline__ float prep(float x) { return x; }
  static __device__ __forceinline__ float combine(float a, float b) { return a + b; }
};
struct OpSumSq {
  static __device__ __forceinline__ float identity() { return 0.f; }
  static __device__ __forceinline__ float prep(float x) { return x * x; }
  static __device__ __forceinline__ float combine(float a, float b) { return a + b; }
};
struct OpMax {
  static __device__ __forceinline__ float identity() { return __int_as_float(0xff800000); }  // -inf
  static __device__ __forceinline__ float prep(float x) { return x; }
  static __device__ __forceinline__ float combine(float a, float b) { return (a > b || a != a) ? a : b; }
};
struct OpMin {
  static __device__ __forceinline__ float identity() { return __int_as_float(0x7f800000); }  // +inf
  static __device__ __forceinline__ float prep(float x) { return x; }
  static __device__ __forceinline__ float combine(float a, float b) { return (a < b || a != a) ? a : b; }
};

// ---------------------------------------------------------------------------
// Reduction building blocks.  Every tree below has a fixed shape, so a given
// input always produces the same bits.
// ---------------------------------------------------------------------------

template <typename Op>
__device__ __forceinline__ float reduce4(float4 v) {
  return Op::combine(Op::combine(Op::prep(v.x), Op::prep(v.y)), Op::combine(Op::prep(v.z), Op::prep(v.w)));
}

// Pairwise reduction of a small register array (values already prepped).
template <typename Op, int N>
__device__ __forceinline__ float tree_reduce(const float* v) {
  if constexpr (N == 1) {
    return v[0];
  } else {
    constexpr int H = N / 2;
    return Op::combine(tree_reduce<Op, H>(v), tree_reduce<Op, N - H>(v + H));
  }
}
template <int N>
__device__ __forceinline__ float tree_sum(const float* v) { return tree_reduce<OpSum, N>(v); }

// Warp reduction: lane 0 receives the reduction of v over the 32 lanes.
template <typename Op>
__device__ __forceinline__ float warp_reduce(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = Op::combine(v, __shfl_down_sync(kFullMask, v, o));
  return v;
}

// Block reduction for NT threads (NT a multiple of 32, at most 1024).  `sh`
// holds NT/32 floats.  The result is valid in thread 0.  The caller must place
// a __syncthreads() between two uses of the same `sh`.
template <typename Op, int NT>
__device__ __forceinline__ float block_reduce(float v, float* sh) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  v = warp_reduce<Op>(v);
  if constexpr (NW == 1) {
    return v;
  } else {
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    float r = Op::identity();
    if (warp == 0) {
      r = lane < NW ? sh[lane] : Op::identity();
#pragma unroll
      for (int o = NW / 2; o > 0; o >>= 1) r = Op::combine(r, __shfl_down_sync(kFullMask, r, o));
    }
    return r;
  }
}
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* sh) { return block_reduce<OpSum, NT>(v, sh); }

// Three-level accumulator.  A plain running fp32 sum over m terms has an
// addition chain of length m, and its worst-case rounding error grows with m.
// Folding the running value into a second, then a third register every K
// terms keeps every chain at most K + K + m/K^2 long, at the cost of two extra
// combines per K terms.  The fold points depend only on the number of terms,
// so the result is deterministic.  (For max and min the folds change nothing.)
template <int K, typename Op = OpSum>
struct BlockedAcc {
  float lo = Op::identity(), mid = Op::identity(), hi = Op::identity();
  int n_lo = 0, n_mid = 0;
  __device__ __forceinline__ void add(float v) {
    lo = Op::combine(lo, v);
    if (++n_lo == K) {
      mid = Op::combine(mid, lo);
      lo = Op::identity();
      n_lo = 0;
      if (++n_mid == K) {
        hi = Op::combine(hi, mid);
        mid = Op::identity();
        n_mid = 0;
      }
    }
  }
  __device__ __forceinline__ float total() const { return Op::combine(hi, Op::combine(mid, lo)); }
};

// Running sum of tile totals: level 0 takes 32 tile totals, each higher level
// 32 folds of the one below, the top one term per 32^4 tiles; hi holds the
// levels above 0, so base() is one addition.
template <int VEC>
struct TileCarry {
  float lv[5][VEC];
  float hi[VEC];
  int n0 = 0, n1 = 0, n2 = 0, n3 = 0;
  __device__ __forceinline__ explicit TileCarry(const float (&init)[VEC]) {
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
#pragma unroll
      for (int k = 0; k < 4; ++k) lv[k][c] = 0.f;
      lv[4][c] = hi[c] = init[c];
    }
  }
  __device__ __forceinline__ void fold(int k) {
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
      lv[k + 1][c] += lv[k][c];
      lv[k][c] = 0.f;
    }
  }
  __device__ __forceinline__ void add(const float (&t)[VEC]) {
#pragma unroll
    for (int c = 0; c < VEC; ++c) lv[0][c] += t[c];
    if (++n0 < 32) return;
    n0 = 0;
    fold(0);
    if (++n1 == 32) {
      n1 = 0;
      fold(1);
      if (++n2 == 32) {
        n2 = 0;
        fold(2);
        if (++n3 == 32) {
          n3 = 0;
          fold(3);
        }
      }
    }
#pragma unroll
    for (int c = 0; c < VEC; ++c) hi[c] = ((lv[4][c] + lv[3][c]) + lv[2][c]) + lv[1][c];
  }
  __device__ __forceinline__ float base(int c) const { return hi[c] + lv[0][c]; }
};

// Output epilogue: the mean divides by the element count (in double, then
// rounds once to fp32); the Euclidean norm takes the square root of the sum
// of squares (IEEE, correctly rounded).
__device__ __forceinline__ float finish(float v, int epi, int64_t count) {
  if (epi == kEpiMean) return (float)((double)v / (double)count);
  if (epi == kEpiSqrt) return sqrtf(v);
  return v;
}

}  // namespace lr
