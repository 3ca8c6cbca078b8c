// lr_rows_short.cu -- cumulative sums and reductions of many short rows
// (inner == 1, N up to kShortRowMax).
//
// One block per row would leave most of its threads idle and pay a whole
// tile's work for a few hundred bytes.  Instead a block stages a chunk of
// whole rows (contiguous in memory; the host sizes it and starts every chunk
// on a 128-byte boundary where the rows allow) in shared memory with
// coalesced loads, scans or reduces every row there, and (scans) stores the
// chunk back with coalesced stores.  The blocks run a software pipeline: the
// next chunk's loads are issued into registers before the current chunk is
// processed.  A row is handled by a group of G lanes:
//   G == 1: one thread walks the row in the scan direction;
//   G > 1:  lane g takes the g-th run of L (odd) consecutive elements from
//           the scan's start: a sequential prefix over its run in place,
//           then the sum of the runs before it from a shuffle scan of the
//           run totals across the group, added to each of its outputs.
// Narrow planes ([outer, N, inner] scanned or reduced along N, inner > 1,
// N <= kShortRowMax) take the same kernels with PLANES set: a chunk holds
// whole planes, contiguous in memory, and is staged transposed -- column c of
// plane q becomes the shared-memory row q*inner + c -- so each column is a
// row to the code below, and the store transposes back.
// Every output is a sum over its own terms (an exclusive output leaves its
// own term out of its run's prefix), so nothing is subtracted, and all orders
// are fixed: reruns are bit-identical.  Rows are padded in shared memory so
// that the lanes of a warp hit distinct banks: an odd row stride for G == 1;
// for G > 1 an odd run length (the lanes of a row are L apart) and a row
// stride congruent to L*G modulo 32 (the rows of a warp then cover distinct
// banks too).
#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

// With 16-byte loads (N % 4 == 0) the row stride is a multiple of 4 for every
// group of at least 4 lanes (stride = L*G mod 32, or N itself for G == 32),
// so staging can use 16-byte shared-memory accesses.
template <int G>
constexpr bool kSmem4 = G >= 4;

// Floats of one row, or of one plane (PLANES).
template <bool PLANES>
__device__ __forceinline__ int unit_len(const ShortRowsParams& p) {
  return PLANES ? p.N * p.inner : p.N;
}

// Shared-memory address of flat chunk index e (row r at r*stride).  An
// unpadded chunk (stride == N: one lane per row with N odd) needs no row.
// PLANES: e = (q*N + j)*inner + c lands in row q*inner + c at column j.
template <bool PLANES>
__device__ __forceinline__ float* chunk_slot_raw(const ShortRowsParams& p, float* s, int e) {
  if constexpr (PLANES) {
    const int qj = (int)(((unsigned long long)e * p.magic_inner) >> 32);  // e / inner
    const int c = e - qj * p.inner;
    const int q = (int)(((unsigned long long)qj * p.magic) >> 32);        // plane in the chunk
    return s + (q * p.inner + c) * p.stride + (qj - q * p.N);
  } else {
    if (p.stride == p.N) return s + e;
    const int r = (int)(((unsigned long long)e * p.magic) >> 32);
    return s + r * p.stride + (e - r * p.N);
  }
}
#ifdef LR_DEBUG
// Debug builds: a slot outside the shared buffer is recorded and replaced by
// slot 0 (its contents are then wrong, and reported).
template <bool PLANES>
__device__ __forceinline__ float* chunk_slot(const ShortRowsParams& p, float* s, int e) {
  float* d = chunk_slot_raw<PLANES>(p, s, e);
  return LR_DBG_SHARED(d - s, 1, kShortSmem, d) ? d : s;
}
#else
template <bool PLANES>
__device__ __forceinline__ float* chunk_slot(const ShortRowsParams& p, float* s, int e) {
  return chunk_slot_raw<PLANES>(p, s, e);
}
#endif

// Coalesced stores of a chunk back to memory.  VEC 4 stores 16 bytes at a
// time (rows: N % 4 == 0, a float4 never straddles two rows; planes: N*inner
// % 4 == 0).  SMEM4: 16-byte shared-memory reads (rows whose stride is a
// multiple of 4: see kSmem4); else four 4-byte ones, each from its own slot
// for planes (the four floats of a 16-byte store lie in four columns).
template <int VEC, bool SMEM4, bool PLANES>
__device__ __forceinline__ void stage_out(const ShortRowsParams& p, float* s, float* dst, int ne) {
  const int t = threadIdx.x;
  if constexpr (VEC == kShortLd4) {
#pragma unroll 4
    for (int e = 4 * t; e < ne; e += 4 * kShortThreads) {
      if constexpr (PLANES) {
        st_stream4(dst + e, make_float4(*chunk_slot<true>(p, s, e), *chunk_slot<true>(p, s, e + 1),
                                        *chunk_slot<true>(p, s, e + 2), *chunk_slot<true>(p, s, e + 3)));
      } else {
        const float* d = chunk_slot<false>(p, s, e);
        if constexpr (SMEM4) st_stream4(dst + e, *reinterpret_cast<const float4*>(d));
        else st_stream4(dst + e, make_float4(d[0], d[1], d[2], d[3]));
      }
    }
  } else {
#pragma unroll 8
    for (int e = t; e < ne; e += kShortThreads) st_stream1(dst + e, *chunk_slot<PLANES>(p, s, e));
  }
}

constexpr int kRegRun = 16;   // elements a lane holds in registers at a time
constexpr int kRunBlock = 8;  // elements per register block of a long run

// Scan the n elements at base[dir*i], i = 0..n-1, in place from zero
// (inclusive, or exclusive: each output leaves its own term out); returns
// their sum.  The additions are the sequential ones: acc += x[0], x[1], ...,
// so an output is at most n - 1 roundings deep (the host keeps walked rows
// to at most 159 elements and lane runs to at most 65).  BLOCKED moves
// kRunBlock elements at a time through registers (all loads of a block
// issued together; the zeros that pad the last block leave acc unchanged),
// which pays where few lanes hold long runs (32-lane groups: rows of
// 500-2048, 0.84-0.86 -> 0.87-0.94 of copy bandwidth); with many groups in
// flight the element-by-element walk, with fewer instructions, is faster
// (rows of 100-256: 0.96 against 0.93).
template <bool BLOCKED>
__device__ __forceinline__ float scan_run(float* base, int dir, int n, bool exclusive) {
  float acc = 0.f;
  if constexpr (!BLOCKED) {
    for (int i = 0; i < n; ++i) {
      const float before = acc;
      acc += base[dir * i];
      base[dir * i] = exclusive ? before : acc;
    }
    return acc;
  }
  for (int i0 = 0; i0 < n; i0 += kRunBlock) {
    float v[kRunBlock];
#pragma unroll
    for (int i = 0; i < kRunBlock; ++i) v[i] = i0 + i < n ? base[dir * (i0 + i)] : 0.f;
#pragma unroll
    for (int i = 0; i < kRunBlock; ++i) {
      const float before = acc;
      acc += v[i];
      v[i] = exclusive ? before : acc;
    }
#pragma unroll
    for (int i = 0; i < kRunBlock; ++i)
      if (i0 + i < n) base[dir * (i0 + i)] = v[i];
  }
  return acc;
}

// base[dir*i] = off + base[dir*i] for i = 0..n-1 (BLOCKED: kRunBlock at a time).
template <bool BLOCKED>
__device__ __forceinline__ void offset_run(float* base, int dir, int n, float off) {
  if constexpr (!BLOCKED) {
    for (int i = 0; i < n; ++i) base[dir * i] = off + base[dir * i];
    return;
  }
  for (int i0 = 0; i0 < n; i0 += kRunBlock) {
    float v[kRunBlock];
#pragma unroll
    for (int i = 0; i < kRunBlock; ++i) v[i] = i0 + i < n ? base[dir * (i0 + i)] : 0.f;
#pragma unroll
    for (int i = 0; i < kRunBlock; ++i)
      if (i0 + i < n) base[dir * (i0 + i)] = off + v[i];
  }
}

// Scan one row in place with G lanes (g = this lane's index in its group).
// G == 1: the lane walks the row in the scan direction.  G > 1: lane g takes
// the g-th run of L consecutive elements counted from the scan's start; the
// sum of the runs before it (an exclusive scan of the run totals across the
// group) is added to each of its prefix sums.  A run of at most kRegRun
// elements stays in registers between its load and its store; a longer one
// is scanned in place first and offset in a second pass (see scan_run).
// Both compute off + (prefix within the run) with the same additions.
// `active` is false for the lanes of a group past the chunk's last row: they
// still take part in the shuffles, with zeros, and touch nothing.
template <int G>
__device__ __forceinline__ void scan_row(float* row, int N, int L, int g, bool active, bool mirror,
                                         bool exclusive) {
  if constexpr (G == 1) {
    if (!active) return;
    scan_run<false>(mirror ? row : row + (N - 1), mirror ? 1 : -1, N, exclusive);
  } else {
    // Element i of run g in memory: g*L + i (forward) or N-1 - (g*L + i)
    // (reverse); positions outside [0, N) belong to no element.
    const int first = g * L;
    const int n_run = active ? max(0, min(L, N - first)) : 0;
    float* base = mirror ? row + first : row + (N - 1 - first);
    const int dir = mirror ? 1 : -1;
    const auto offset_of = [&](float total) {
      float incl = total;  // prefix of the run totals over lanes 0..g
#pragma unroll
      for (int d = 1; d < G; d <<= 1) {
        const float o = __shfl_up_sync(kFullMask, incl, d, G);
        if (g >= d) incl += o;
      }
      const float off = __shfl_up_sync(kFullMask, incl, 1, G);  // the runs before this one
      return g == 0 ? 0.f : off;
    };
    if (L <= kRegRun) {  // the same for every lane of the warp
      float v[kRegRun];
#pragma unroll
      for (int i = 0; i < kRegRun; ++i) v[i] = i < n_run ? base[dir * i] : 0.f;
      float total = 0.f;
#pragma unroll
      for (int i = 0; i < kRegRun; ++i) total += v[i];
      const float off = offset_of(total);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < kRegRun; ++i) {
        const float before = acc;
        acc += v[i];
        v[i] = off + (exclusive ? before : acc);
      }
#pragma unroll
      for (int i = 0; i < kRegRun; ++i)
        if (i < n_run) base[dir * i] = v[i];
    } else {
      const float off = offset_of(scan_run<(G == 32)>(base, dir, n_run, exclusive));
      offset_run<(G == 32)>(base, dir, n_run, off);
    }
  }
}

// The software pipeline: a thread loads its share of the first kShortChunk
// floats of chunk c + gridDim.x into registers (kPrefetch loads of 16 or 4
// bytes) while chunk c is being processed, and writes them to shared memory
// when that chunk is staged.  A longer chunk loads the rest at staging.
template <int VEC>
struct ChunkRegs {  // kShortLd4
  static constexpr int kWidth = 4;
  static constexpr int kPrefetch = kShortChunk / (4 * kShortThreads);  // 6
  float4 v[kPrefetch];
};
template <>
struct ChunkRegs<kShortLd1> {
  static constexpr int kWidth = 1;
  static constexpr int kPrefetch = kShortChunk / kShortThreads;  // 24
  float v[kPrefetch];
};
static_assert(ChunkRegs<kShortLd4>::kPrefetch * 4 * kShortThreads == kShortChunk &&
                  ChunkRegs<kShortLd1>::kPrefetch * kShortThreads == kShortChunk,
              "a prefetch covers kShortChunk floats");

// One load at chunk index e of src: 16 bytes or 4.
template <int VEC>
__device__ __forceinline__ auto ld_chunk(const float* src, int e) {
  if constexpr (VEC == kShortLd4) return ld_stream4(src + e);
  else return ld_stream1(src + e);
}

template <int VEC, bool PLANES>
__device__ __forceinline__ void prefetch_chunk(const ShortRowsParams& p, int64_t c, ChunkRegs<VEC>& f) {
  const int64_t r0 = c * p.rows_per_chunk;
  const int ne = (int)min((int64_t)p.rows_per_chunk, p.rows - r0) * unit_len<PLANES>(p);
  const float* src = p.x + r0 * unit_len<PLANES>(p);
#pragma unroll
  for (int k = 0; k < ChunkRegs<VEC>::kPrefetch; ++k) {
    const int e = ChunkRegs<VEC>::kWidth * (threadIdx.x + k * kShortThreads);
    if (e < ne) f.v[k] = ld_chunk<VEC>(src, e);
  }
}

// One load's worth (chunk index e) into shared memory: a 16-byte store
// (SMEM4), four 4-byte ones (each to its own slot for planes), or one float.
template <int VEC, bool SMEM4, bool PLANES>
__device__ __forceinline__ void put(const ShortRowsParams& p, float* s, int e, float4 v) {
  if constexpr (PLANES) {
    *chunk_slot<true>(p, s, e) = v.x;
    *chunk_slot<true>(p, s, e + 1) = v.y;
    *chunk_slot<true>(p, s, e + 2) = v.z;
    *chunk_slot<true>(p, s, e + 3) = v.w;
  } else {
    float* d = chunk_slot<false>(p, s, e);
    if constexpr (SMEM4) {
      *reinterpret_cast<float4*>(d) = v;
    } else {
      d[0] = v.x;
      d[1] = v.y;
      d[2] = v.z;
      d[3] = v.w;
    }
  }
}
template <int VEC, bool SMEM4, bool PLANES>
__device__ __forceinline__ void put(const ShortRowsParams& p, float* s, int e, float v) {
  *chunk_slot<PLANES>(p, s, e) = v;
}

// Stage the ne floats of the chunk starting at row (or plane) r0 from the
// prefetched registers, plus the rest of a chunk longer than the prefetch.
template <int G, int VEC, bool PLANES>
__device__ __forceinline__ void stage_chunk(const ShortRowsParams& p, float* s, int64_t r0, int ne,
                                            const ChunkRegs<VEC>& f) {
  constexpr int W = ChunkRegs<VEC>::kWidth;
  const int t = threadIdx.x;
#pragma unroll
  for (int k = 0; k < ChunkRegs<VEC>::kPrefetch; ++k) {
    const int e = W * (t + k * kShortThreads);
    if (e < ne) put<VEC, kSmem4<G>, PLANES>(p, s, e, f.v[k]);
  }
  const float* src = p.x + r0 * unit_len<PLANES>(p);
#pragma unroll 2
  for (int e = W * (t + ChunkRegs<VEC>::kPrefetch * kShortThreads); e < ne; e += W * kShortThreads)
    put<VEC, kSmem4<G>, PLANES>(p, s, e, ld_chunk<VEC>(src, e));
}

template <int G, int VEC, bool PLANES>
__global__ void __launch_bounds__(kShortThreads, 7) k_rscan_short(ShortRowsParams p) {
  pdl_begin();
  __shared__ __align__(16) float s[kShortSmem];
  const int t = threadIdx.x;
  const int gi = t / G;  // this thread's group
  const int g = t % G;   // its lane in the group
  constexpr int kGroups = kShortThreads / G;
  const bool mirror = (p.flags & kScanMirror) != 0;
  const bool exclusive = (p.flags & kScanExclusive) != 0;
  const int64_t chunks = (p.rows + p.rows_per_chunk - 1) / p.rows_per_chunk;
  const int inner = PLANES ? p.inner : 1;
  ChunkRegs<VEC> f;
  if (blockIdx.x < chunks) prefetch_chunk<VEC, PLANES>(p, blockIdx.x, f);
  for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x) {
    const int64_t r0 = c * p.rows_per_chunk;
    const int nr = (int)min((int64_t)p.rows_per_chunk, p.rows - r0) * inner;  // rows in shared memory
    const int ne = nr * p.N;
    stage_chunk<G, VEC, PLANES>(p, s, r0, ne, f);
    __syncthreads();
    if (c + gridDim.x < chunks) prefetch_chunk<VEC, PLANES>(p, c + gridDim.x, f);
    // Whole warps stay in the loop (the groups' shuffles), so the bound is
    // the same for every thread.
    for (int rb = 0; rb < nr; rb += kGroups) {
      const int r = rb + gi;
      float* row = s + (r < nr ? r : 0) * p.stride;
      // Debug builds: a row reaching outside the shared buffer is recorded and skipped.
      const bool in_smem = LR_DBG_SHARED(row - s, p.N, kShortSmem, row);
      scan_row<G>(row, p.N, p.run_len, g, r < nr && in_smem, mirror, exclusive);
    }
    __syncthreads();
    stage_out<VEC, kSmem4<G>, PLANES>(p, s, p.y + r0 * unit_len<PLANES>(p), ne);
    __syncthreads();  // the next chunk overwrites s
  }
}

// Reductions of many short rows: the same chunks and lane groups.  Lane g of
// a row's group combines its run (elements g*L .. g*L+L-1 in order), the
// group's lanes are then combined by a fixed shuffle tree, and lane 0 writes
// the row's result (with the epilogue: mean or square root).  p.y is the
// output (one float per row) and p.flags the epilogue.
template <int G, int VEC, typename Op, bool PLANES>
__global__ void __launch_bounds__(kShortThreads, 7) k_reduce_short(ShortRowsParams p) {
  pdl_begin();
  __shared__ __align__(16) float s[kShortSmem];
  const int t = threadIdx.x;
  const int gi = t / G;
  const int g = t % G;
  constexpr int kGroups = kShortThreads / G;
  const int64_t chunks = (p.rows + p.rows_per_chunk - 1) / p.rows_per_chunk;
  const int inner = PLANES ? p.inner : 1;
  ChunkRegs<VEC> f;
  if (blockIdx.x < chunks) prefetch_chunk<VEC, PLANES>(p, blockIdx.x, f);
  for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x) {
    const int64_t r0 = c * p.rows_per_chunk;
    const int nr = (int)min((int64_t)p.rows_per_chunk, p.rows - r0) * inner;  // rows in shared memory
    stage_chunk<G, VEC, PLANES>(p, s, r0, nr * p.N, f);
    __syncthreads();
    if (c + gridDim.x < chunks) prefetch_chunk<VEC, PLANES>(p, c + gridDim.x, f);
    for (int rb = 0; rb < nr; rb += kGroups) {
      const int r = rb + gi;
      const float* row = s + (r < nr ? r : 0) * p.stride;
      const bool active = r < nr && LR_DBG_SHARED(row - s, p.N, kShortSmem, row);
      const int first = G == 1 ? 0 : g * p.run_len;
      const int n_run = active ? max(0, min(G == 1 ? p.N : p.run_len, p.N - first)) : 0;
      // Whole blocks of kRegRun elements, each combined by a fixed tree, then
      // the remaining elements, all folded in order: a row of up to 128
      // elements is at most log2(kRegRun) + 8 + 15 roundings deep.
      float v = Op::identity();
      const float* rp = row + first;
      int i0 = 0;
      for (; i0 + kRegRun <= n_run; i0 += kRegRun) {
        float a[kRegRun];
#pragma unroll
        for (int i = 0; i < kRegRun; ++i) a[i] = Op::prep(rp[i0 + i]);
        v = Op::combine(v, tree_reduce<Op, kRegRun>(a));
      }
#pragma unroll 4
      for (; i0 < n_run; ++i0) v = Op::combine(v, Op::prep(rp[i0]));
      if constexpr (G > 1) {
#pragma unroll
        for (int d = G / 2; d > 0; d >>= 1) v = Op::combine(v, __shfl_down_sync(kFullMask, v, d, G));
      }
      if (active && g == 0) st_plain(p.y + r0 * inner + r, finish(v, p.flags, p.N));  // output (plane, column)
    }
    __syncthreads();  // the next chunk overwrites s
  }
}

template <int G, typename Op, bool PLANES>
cudaError_t launch_reduce_gp(int vec, const ShortRowsParams& p, int64_t grid, cudaStream_t s) {
  if (vec == kShortLd4) {
    launch_pdl(k_reduce_short<G, kShortLd4, Op, PLANES>, dim3((unsigned)grid), kShortThreads, 0, s, p);
  } else {
    launch_pdl(k_reduce_short<G, kShortLd1, Op, PLANES>, dim3((unsigned)grid), kShortThreads, 0, s, p);
  }
  return cudaGetLastError();
}
template <int G, typename Op>
cudaError_t launch_reduce_g(int vec, const ShortRowsParams& p, int64_t grid, cudaStream_t s) {
  return p.inner > 1 ? launch_reduce_gp<G, Op, true>(vec, p, grid, s) : launch_reduce_gp<G, Op, false>(vec, p, grid, s);
}

template <typename Op>
cudaError_t launch_reduce_op(int lanes, int vec, const ShortRowsParams& p, int64_t grid, cudaStream_t s) {
  switch (lanes) {
    case 1: return launch_reduce_g<1, Op>(vec, p, grid, s);
    case 2: return launch_reduce_g<2, Op>(vec, p, grid, s);
    case 4: return launch_reduce_g<4, Op>(vec, p, grid, s);
    case 8: return launch_reduce_g<8, Op>(vec, p, grid, s);
    case 16: return launch_reduce_g<16, Op>(vec, p, grid, s);
    case 32: return launch_reduce_g<32, Op>(vec, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int G, bool PLANES>
cudaError_t launch_gp(int vec, const ShortRowsParams& p, int64_t grid, cudaStream_t s) {
  if (vec == kShortLd4) {
    launch_pdl(k_rscan_short<G, kShortLd4, PLANES>, dim3((unsigned)grid), kShortThreads, 0, s, p);
  } else {
    launch_pdl(k_rscan_short<G, kShortLd1, PLANES>, dim3((unsigned)grid), kShortThreads, 0, s, p);
  }
  return cudaGetLastError();
}
template <int G>
cudaError_t launch_g(int vec, const ShortRowsParams& p, int64_t grid, cudaStream_t s) {
  return p.inner > 1 ? launch_gp<G, true>(vec, p, grid, s) : launch_gp<G, false>(vec, p, grid, s);
}

}  // namespace

cudaError_t launch_rscan_short(int lanes, int vec, const ShortRowsParams& p, int64_t grid, cudaStream_t s) {
  switch (lanes) {
    case 1: return launch_g<1>(vec, p, grid, s);
    case 2: return launch_g<2>(vec, p, grid, s);
    case 4: return launch_g<4>(vec, p, grid, s);
    case 8: return launch_g<8>(vec, p, grid, s);
    case 16: return launch_g<16>(vec, p, grid, s);
    case 32: return launch_g<32>(vec, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_reduce_short(int op, int lanes, int vec, const ShortRowsParams& p, int64_t grid, cudaStream_t s) {
  switch (op) {
    case kOpSum: return launch_reduce_op<OpSum>(lanes, vec, p, grid, s);
    case kOpSumSq: return launch_reduce_op<OpSumSq>(lanes, vec, p, grid, s);
    case kOpMax: return launch_reduce_op<OpMax>(lanes, vec, p, grid, s);
    case kOpMin: return launch_reduce_op<OpMin>(lanes, vec, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

int occupancy_rscan_short() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_rscan_short<32, kShortLd4, false>, kShortThreads, 0) !=
      cudaSuccess)
    return 0;
  return n;
}

}  // namespace lr
