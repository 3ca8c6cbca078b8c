// lr_rows_short.cu -- cumulative sums and reductions of many short rows
// (inner == 1, N up to kShortRowMax).
//
// One block per row would leave most of its threads idle and pay a whole
// tile's work for a few hundred bytes.  Instead a block stages a chunk of
// whole rows (contiguous in memory; the host sizes it and starts every chunk
// on a 128-byte boundary where the rows allow) in shared memory with
// coalesced loads, scans or reduces every row there, and (scans) stores the
// chunk back with coalesced stores.  With 16-byte loads the blocks run a
// software pipeline: the next chunk's loads are issued into registers before
// the current chunk is processed.  A row is handled by a group of G lanes:
//   G == 1: one thread walks the row in the scan direction;
//   G > 1:  lane g takes the g-th run of L (odd) consecutive elements from
//           the scan's start: a sequential prefix over its run in place,
//           then the sum of the runs before it from a shuffle scan of the
//           run totals across the group, added to each of its outputs.
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

// Coalesced stores of a chunk back to memory.  VEC 4 stores 16 bytes at a
// time (N % 4 == 0: a float4 never straddles two rows).  SMEM4: 16-byte
// shared-memory reads (the row stride is a multiple of 4: see kSmem4); else
// four 4-byte ones.
template <int VEC, bool SMEM4>
__device__ __forceinline__ void stage_out(const ShortRowsParams& p, const float* s, float* dst, int ne) {
  const int t = threadIdx.x;
  if constexpr (VEC == 4) {
#pragma unroll 4
    for (int e = 4 * t; e < ne; e += 4 * kShortThreads) {
      const int r = (int)(((unsigned long long)e * p.magic) >> 32);
      const float* d = s + r * p.stride + (e - r * p.N);
      if constexpr (SMEM4) st_stream4(dst + e, *reinterpret_cast<const float4*>(d));
      else st_stream4(dst + e, make_float4(d[0], d[1], d[2], d[3]));
    }
  } else {
#pragma unroll 8
    for (int e = t; e < ne; e += kShortThreads) {
      const int r = (int)(((unsigned long long)e * p.magic) >> 32);
      st_stream1(dst + e, s[r * p.stride + (e - r * p.N)]);
    }
  }
}

constexpr int kRegRun = 16;  // elements a lane holds in registers at a time

// Scan one row in place with G lanes (g = this lane's index in its group).
// G == 1: the lane walks the row in the scan direction.  G > 1: lane g takes
// the g-th run of L consecutive elements counted from the scan's start; the
// sum of the runs before it (an exclusive scan of the run totals across the
// group) is added to each of its prefix sums.  A run of at most kRegRun
// elements stays in registers between its load and its store; a longer one
// is scanned in place first and offset in a second pass.  Both compute
// off + (prefix within the run) with the same additions.
// `active` is false for the lanes of a group past the chunk's last row: they
// still take part in the shuffles, with zeros, and touch nothing.
template <int G>
__device__ __forceinline__ void scan_row(float* row, int N, int L, int g, bool active, bool mirror,
                                         bool exclusive) {
  if constexpr (G == 1) {
    if (!active) return;
    float acc = 0.f;
    const int dir = mirror ? 1 : -1;
    float* p0 = mirror ? row : row + (N - 1);
    for (int i = 0; i < N; ++i) {
      const float before = acc;
      acc += p0[dir * i];
      p0[dir * i] = exclusive ? before : acc;
    }
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
      float acc = 0.f;
      for (int i = 0; i < n_run; ++i) {
        const float before = acc;
        acc += base[dir * i];
        base[dir * i] = exclusive ? before : acc;
      }
      const float off = offset_of(acc);
      for (int i = 0; i < n_run; ++i) base[dir * i] = off + base[dir * i];
    }
  }
}

// The software pipeline: a thread loads its share of the first kShortChunk
// floats of chunk c + gridDim.x into registers (kPrefetch loads of VEC
// floats) while chunk c is being processed, and writes them to shared memory
// when that chunk is staged.  A longer chunk loads the rest at staging.
template <int VEC>
struct ChunkRegs;
template <>
struct ChunkRegs<4> {
  static constexpr int kPrefetch = kShortChunk / (4 * kShortThreads);  // 6
  float4 v[kPrefetch];
};
template <>
struct ChunkRegs<1> {
  static constexpr int kPrefetch = kShortChunk / kShortThreads;  // 24
  float v[kPrefetch];
};
static_assert(ChunkRegs<4>::kPrefetch * 4 * kShortThreads == kShortChunk &&
                  ChunkRegs<1>::kPrefetch * kShortThreads == kShortChunk,
              "a prefetch covers kShortChunk floats");

template <int VEC>
__device__ __forceinline__ auto ld_vec(const float* p) {
  if constexpr (VEC == 4) return ld_stream4(p);
  else return ld_stream1(p);
}

template <int VEC>
__device__ __forceinline__ void prefetch_chunk(const ShortRowsParams& p, int64_t c, ChunkRegs<VEC>& f) {
  const int64_t r0 = c * p.rows_per_chunk;
  const int ne = (int)min((int64_t)p.rows_per_chunk, p.rows - r0) * p.N;
  const float* src = p.x + r0 * p.N;
#pragma unroll
  for (int k = 0; k < ChunkRegs<VEC>::kPrefetch; ++k) {
    const int e = VEC * (threadIdx.x + k * kShortThreads);
    if (e < ne) f.v[k] = ld_vec<VEC>(src + e);
  }
}

// Shared-memory address of flat chunk index e (row r at r*stride).
__device__ __forceinline__ float* chunk_slot(const ShortRowsParams& p, float* s, int e) {
  const int r = (int)(((unsigned long long)e * p.magic) >> 32);
  return s + r * p.stride + (e - r * p.N);
}

// One load's worth of a chunk into shared memory: a 16-byte store (SMEM4),
// four 4-byte ones, or one float.
template <bool SMEM4>
__device__ __forceinline__ void put(float* d, float4 v) {
  if constexpr (SMEM4) {
    *reinterpret_cast<float4*>(d) = v;
  } else {
    d[0] = v.x;
    d[1] = v.y;
    d[2] = v.z;
    d[3] = v.w;
  }
}
template <bool SMEM4>
__device__ __forceinline__ void put(float* d, float v) {
  *d = v;
}

// Stage the ne floats of the chunk starting at row r0 from the prefetched
// registers, plus the rest of a chunk longer than the prefetch.
template <int G, int VEC>
__device__ __forceinline__ void stage_chunk(const ShortRowsParams& p, float* s, int64_t r0, int ne,
                                            const ChunkRegs<VEC>& f) {
  const int t = threadIdx.x;
#pragma unroll
  for (int k = 0; k < ChunkRegs<VEC>::kPrefetch; ++k) {
    const int e = VEC * (t + k * kShortThreads);
    if (e < ne) put<kSmem4<G>>(chunk_slot(p, s, e), f.v[k]);
  }
  const float* src = p.x + r0 * p.N;
#pragma unroll 2
  for (int e = VEC * (t + ChunkRegs<VEC>::kPrefetch * kShortThreads); e < ne; e += VEC * kShortThreads)
    put<kSmem4<G>>(chunk_slot(p, s, e), ld_vec<VEC>(src + e));
}

template <int G, int VEC>
__global__ void __launch_bounds__(kShortThreads, 7) k_rscan_short(ShortRowsParams p) {
  __shared__ __align__(16) float s[kShortSmem];
  const int t = threadIdx.x;
  const int gi = t / G;  // this thread's group
  const int g = t % G;   // its lane in the group
  constexpr int kGroups = kShortThreads / G;
  const bool mirror = (p.flags & kScanMirror) != 0;
  const bool exclusive = (p.flags & kScanExclusive) != 0;
  const int64_t chunks = (p.rows + p.rows_per_chunk - 1) / p.rows_per_chunk;
  ChunkRegs<VEC> f;
  if (blockIdx.x < chunks) prefetch_chunk<VEC>(p, blockIdx.x, f);
  for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x) {
    const int64_t r0 = c * p.rows_per_chunk;
    const int nr = (int)min((int64_t)p.rows_per_chunk, p.rows - r0);
    const int ne = nr * p.N;
    stage_chunk<G, VEC>(p, s, r0, ne, f);
    __syncthreads();
    if (c + gridDim.x < chunks) prefetch_chunk<VEC>(p, c + gridDim.x, f);
    // Whole warps stay in the loop (the groups' shuffles), so the bound is
    // the same for every thread.
    for (int rb = 0; rb < nr; rb += kGroups) {
      const int r = rb + gi;
      scan_row<G>(s + (r < nr ? r : 0) * p.stride, p.N, p.run_len, g, r < nr, mirror, exclusive);
    }
    __syncthreads();
    stage_out<VEC, kSmem4<G>>(p, s, p.y + r0 * p.N, ne);
    __syncthreads();  // the next chunk overwrites s
  }
}

// Reductions of many short rows: the same chunks and lane groups.  Lane g of
// a row's group combines its run (elements g*L .. g*L+L-1 in order), the
// group's lanes are then combined by a fixed shuffle tree, and lane 0 writes
// the row's result (with the epilogue: mean or square root).  p.y is the
// output (one float per row) and p.flags the epilogue.
template <int G, int VEC, typename Op>
__global__ void __launch_bounds__(kShortThreads, 7) k_reduce_short(ShortRowsParams p) {
  __shared__ __align__(16) float s[kShortSmem];
  const int t = threadIdx.x;
  const int gi = t / G;
  const int g = t % G;
  constexpr int kGroups = kShortThreads / G;
  const int64_t chunks = (p.rows + p.rows_per_chunk - 1) / p.rows_per_chunk;
  ChunkRegs<VEC> f;
  if (blockIdx.x < chunks) prefetch_chunk<VEC>(p, blockIdx.x, f);
  for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x) {
    const int64_t r0 = c * p.rows_per_chunk;
    const int nr = (int)min((int64_t)p.rows_per_chunk, p.rows - r0);
    stage_chunk<G, VEC>(p, s, r0, nr * p.N, f);
    __syncthreads();
    if (c + gridDim.x < chunks) prefetch_chunk<VEC>(p, c + gridDim.x, f);
    for (int rb = 0; rb < nr; rb += kGroups) {
      const int r = rb + gi;
      const bool active = r < nr;
      const float* row = s + (active ? r : 0) * p.stride;
      const int first = G == 1 ? 0 : g * p.run_len;
      const int n_run = active ? max(0, min(G == 1 ? p.N : p.run_len, p.N - first)) : 0;
      float v = Op::identity();
      for (int i0 = 0; i0 < n_run; i0 += kRegRun) {
        float a[kRegRun];
#pragma unroll
        for (int i = 0; i < kRegRun; ++i) a[i] = i0 + i < n_run ? Op::prep(row[first + i0 + i]) : Op::identity();
#pragma unroll
        for (int i = 0; i < kRegRun; ++i) v = Op::combine(v, a[i]);
      }
      if constexpr (G > 1) {
#pragma unroll
        for (int d = G / 2; d > 0; d >>= 1) v = Op::combine(v, __shfl_down_sync(kFullMask, v, d, G));
      }
      if (active && g == 0) p.y[r0 + r] = finish(v, p.flags, p.N);
    }
    __syncthreads();  // the next chunk overwrites s
  }
}

template <int G, typename Op>
cudaError_t launch_reduce_g(int vec, const ShortRowsParams& p, int64_t grid, cudaStream_t s) {
  if (vec == 4) k_reduce_short<G, 4, Op><<<dim3((unsigned)grid), kShortThreads, 0, s>>>(p);
  else k_reduce_short<G, 1, Op><<<dim3((unsigned)grid), kShortThreads, 0, s>>>(p);
  return cudaGetLastError();
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

template <int G>
cudaError_t launch_g(int vec, const ShortRowsParams& p, int64_t grid, cudaStream_t s) {
  if (vec == 4) k_rscan_short<G, 4><<<dim3((unsigned)grid), kShortThreads, 0, s>>>(p);
  else k_rscan_short<G, 1><<<dim3((unsigned)grid), kShortThreads, 0, s>>>(p);
  return cudaGetLastError();
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
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_rscan_short<32, 4>, kShortThreads, 0) != cudaSuccess) return 0;
  return n;
}

}  // namespace lr
