// lr_narrow.cu -- reductions and cumulative sums along a strided axis whose
// rows are narrow: x is [outer, N, inner] with inner at most 256 column groups
// of VEC floats (the library routes up to 256 scalar or 128 float4 columns
// here) (sm_103a).
//
// The wide-row kernels put a warp across 32*VEC adjacent columns and loop down
// the axis (POPCORNBENCH trace l1_p47: coalesced across the contiguous inner
// dim).  With a narrow row most of those lanes would hold no column.  Here the
// [N, inner] plane of each o is read as the contiguous array it is: a thread
// owns one group of VEC adjacent columns, and the block's threads span G
// consecutive rows (G = 256 / threads per row), so one block-wide step reads
// G*inner consecutive floats while every thread keeps its column.
//
// Accuracy is by construction, as elsewhere: blocked accumulators and fixed
// trees (reduction), per-thread runs of U rows, a warp shuffle scan over the
// row groups, warp totals in a fixed order and the blocked tile carry (scan);
// no output subtracts anything.
#include "lr_contig.cuh"
#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

constexpr int kNW = kThreads / 32;

template <typename K>
int occupancy_of(K kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess) return 0;
  return n;
}

template <int VEC>
__device__ __forceinline__ void load_vec(float (&v)[VEC], const float* p) {
  if constexpr (VEC == 4) {
    const float4 f = ld_stream4(p);
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
  } else {
    v[0] = ld_stream1(p);
  }
}

template <int VEC>
__device__ __forceinline__ void store_vec(float* p, const float (&v)[VEC]) {
  if constexpr (VEC == 4)
    st_stream4(p, make_float4(v[0], v[1], v[2], v[3]));
  else
    st_stream1(p, v[0]);
}

// Combine the per-row-group values sh[g * inner + c] (g < G) into sh[c] with a
// fixed pairwise tree over g (G padded to a power of two with nothing).
template <typename Op>
__device__ __forceinline__ void combine_groups(float* sh, int G, int64_t inner) {
  int gp = 1;
  while (gp < G) gp <<= 1;
  const int n = G * (int)inner;
  for (int h = gp >> 1; h >= 1; h >>= 1) {
    const int span = h * (int)inner;
    for (int e = threadIdx.x; e < span; e += kThreads)
      if (e + span < n) sh[e] = Op::combine(sh[e], sh[e + span]);
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Reduction: block (o, slice s) covers rows [s*rows_per_split, ...) of plane
// o; thread (g, cg) reads rows g, g + G, g + 2G, ... of its columns, U rows in
// flight, and keeps a blocked accumulator per column.  The G row groups are
// combined by a tree in shared memory; with one slice that is the output,
// otherwise the slice's column values go to partials and the last block of o
// (integer ticket) combines the slices: its threads take slices g, g + G', ...
// and a second tree joins them.
// ---------------------------------------------------------------------------
template <int VEC, int U, typename Op>
__global__ void __launch_bounds__(kThreads) k_reduce_narrow(NarrowParams p) {
  pdl_begin();
  __shared__ __align__(16) float sh[kThreads * VEC];
  __shared__ int am_last;
  const int64_t inner = p.inner;
  const int tpr = (int)(inner / VEC);  // threads per row; inner % VEC == 0
  const int G = kThreads / tpr;
  const int g = threadIdx.x / tpr;
  const int cg = threadIdx.x - g * tpr;
  const bool active = g < G;
  const int64_t s = blockIdx.x % p.splits;
  const int64_t o = blockIdx.x / p.splits;
  const int64_t r0 = s * p.rows_per_split;
  const int64_t r1 = min(r0 + p.rows_per_split, p.reduce);

  float res[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) res[c] = Op::identity();
  if (active) {
    const float* xc = p.x + o * p.reduce * inner + cg * VEC;
    BlockedAcc<kFold, Op> acc[VEC];
    int64_t r = r0 + g;
    for (; r + (int64_t)(U - 1) * G < r1; r += (int64_t)U * G) {
      float q[U][VEC];
#pragma unroll
      for (int u = 0; u < U; ++u) load_vec<VEC>(q[u], xc + (r + (int64_t)u * G) * inner);
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        float e[U];
#pragma unroll
        for (int u = 0; u < U; ++u) e[u] = Op::prep(q[u][c]);
        acc[c].add(tree_reduce<Op, U>(e));
      }
    }
    for (; r < r1; r += G) {
      float q[VEC];
      load_vec<VEC>(q, xc + r * inner);
#pragma unroll
      for (int c = 0; c < VEC; ++c) acc[c].add(Op::prep(q[c]));
    }
#pragma unroll
    for (int c = 0; c < VEC; ++c) res[c] = acc[c].total();
#pragma unroll
    for (int c = 0; c < VEC; ++c) sh[threadIdx.x * VEC + c] = res[c];  // = sh[g * inner + cg*VEC + c]
  }
  __syncthreads();
  combine_groups<Op>(sh, G, inner);

  if (p.splits == 1) {
    if (threadIdx.x < inner) st_plain(p.out + o * inner + threadIdx.x, finish(sh[threadIdx.x], p.epi, p.reduce));
    return;
  }
  float* part = p.partials + o * p.splits * p.part_stride;
  if (threadIdx.x < p.part_stride)  // part_stride >= inner; the padding columns hold nothing
    st_plain(part + s * p.part_stride + threadIdx.x, threadIdx.x < inner ? sh[threadIdx.x] : Op::identity());
  if (p.keep_partials) return;  // the slice values are the result
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = take_count(p.tickets + o);
    am_last = (prev == (unsigned)(p.splits - 1));
    if (am_last) st_plain(p.tickets + o, 0u);  // every other block of o has taken its ticket
  }
  __syncthreads();
  if (!am_last) return;
  __threadfence();
  const int Gs = kThreads / (int)inner;  // slice groups (inner <= 256 here, so Gs >= 1)
  const int gs = threadIdx.x / (int)inner;
  const int c = threadIdx.x - gs * (int)inner;
  float v = Op::identity();
  if (gs < Gs) {
    BlockedAcc<kFold, Op> acc;
    for (int64_t k = gs; k < p.splits; k += Gs) acc.add(ld_cg1(part + k * p.part_stride + c));
    v = acc.total();
  }
  __syncthreads();  // sh was read by the slice writers above
  if (gs < Gs) sh[threadIdx.x] = v;  // = sh[gs * inner + c]
  __syncthreads();
  combine_groups<Op>(sh, Gs, inner);
  if (threadIdx.x < inner) st_plain(p.out + o * inner + threadIdx.x, finish(sh[threadIdx.x], p.epi, p.reduce));
}

// ---------------------------------------------------------------------------
// Cumulative sum: block per (o, segment); tiles of T = G*U rows in scan order.
// Thread (g, cg) owns scan-order rows [g*U, g*U + U) of the tile.  Tiles are
// staged in shared memory, two buffers: while the block scans tile i, its
// threads' cp.async copies bring tile i + 1 in, with the reduction's mapping
// (step k copies physical rows k*G .. k*G + G - 1: contiguous in memory; rows
// outside the segment arrive as zeros).  Each thread scans its U rows in
// shared memory, the row groups are scanned with warp shuffles (groups of a
// warp: stride tpr lanes) and warp totals, results go back to the same places
// and the block stores the tile contiguously.  Row group g's U rows sit at
// g*S, S = U*inner + pad, the pad chosen so that the lanes of one
// shared-memory access hit distinct banks.  tpr = threads per row, inner / VEC
// rounded up to a power of two (<= 256); from tpr = 32 on a row group spans
// whole warps and the groups' totals meet in shared memory instead.  The
// copies run one tile ahead across the block's planes and segments too.
// ---------------------------------------------------------------------------
template <int VEC, int U>
__host__ __device__ constexpr int scan_narrow_cap() {  // floats of one tile buffer, pad included
  return kThreads * U * VEC + (VEC == 4 ? 1024 : 4096);
}

template <int VEC, int U>
__global__ void __launch_bounds__(kThreads) k_scan_narrow(ScanColsParams p) {
  pdl_begin();
  constexpr int kCap = scan_narrow_cap<VEC, U>();
  extern __shared__ __align__(16) float s_dyn[];         // two tile buffers of kCap floats
  __shared__ __align__(16) float s_tot[kThreads * VEC];  // warp totals, or row-group totals
  const int64_t inner = p.inner;
  int tpr = 1;
  while (tpr * VEC < inner) tpr <<= 1;  // <= 256
  const int G = kThreads / tpr;
  const int T = G * U;
  const int pad = (VEC * tpr - (int)((U * inner) & 31) + 32) & 31;
  const int S = U * (int)inner + pad;
  if (G * S > kCap) return;  // unreachable: tpr <= 256 keeps G*S within kCap
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int warp = t >> 5;
  const int g = t / tpr;
  const int cg = t - g * tpr;
  const int col = cg * VEC;
  const bool active = col < inner;      // with VEC == 4, inner % 4 == 0: all four columns
  const bool wide_groups = tpr >= 32;   // a row group spans whole warps
  const int gpw = wide_groups ? 1 : 32 / tpr;
  const int gcols = tpr * VEC;          // row width of the row-group totals
  const int64_t units = p.outer * p.segs;

  struct Unit {
    int64_t lo, len, tiles;
    const float* xo;
    float* yo;
  };
  const auto unit_at = [&](int64_t u) {
    Unit r;
    const int64_t o = u / p.segs;
    r.lo = (u - o * p.segs) * p.seg_len;
    r.len = min(p.seg_len, p.N - r.lo);
    r.tiles = (r.len + T - 1) / T;
    r.xo = p.x + o * p.N * inner + col;
    r.yo = p.y + o * p.N * inner + col;
    return r;
  };
  // Physical rows of tile i: [phys_lo, phys_lo + T) clipped to the segment.
  const auto phys_lo = [&](const Unit& un, int64_t i) {
    return p.reverse ? un.lo + un.len - (i + 1) * T : un.lo + i * T;
  };
  // The tile geometry (G, S, inner) is hidden from the optimiser once per
  // tile (Gt, St, It): otherwise it hoists every row's shared-memory offset
  // out of the tile loop and holds them all in registers.
  const auto issue = [&](float* buf, const Unit& un, int64_t i, int Gt, int St, int It) {
    if (!active) return;
    const int64_t pl = phys_lo(un, i);
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int pr = k * Gt + g;  // tile row; group pr / U, row pr % U within it
      const int64_t row = pl + pr;
      const bool ok = row >= un.lo && row < un.lo + un.len;
      float* d = buf + (pr / U) * St + (pr % U) * It + col;
      const float* src = ok ? un.xo + row * inner : un.xo;
      if constexpr (VEC == 4)
        cp_async16(d, src, ok ? 16u : 0u);
      else
        cp_async4(d, src, ok ? 4u : 0u);
    }
  };
  const auto carry_of = [&](int64_t u) {
    float init[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c)
      init[c] = (p.carry != nullptr && active) ? ld_plain(p.carry + u * p.carry_stride + col + c) : 0.f;
    return TileCarry<VEC>(init);
  };

  int64_t unit = blockIdx.x;
  if (unit >= units) return;
  Unit cu = unit_at(unit);
  TileCarry<VEC> tc = carry_of(unit);
  int cur = 0;
  int64_t i = 0;
  issue(s_dyn, cu, 0, G, S, (int)inner);
  cp_async_commit();
  while (true) {
    int Gt = G, St = S, It = (int)inner;
    asm volatile("" : "+r"(Gt), "+r"(St), "+r"(It));
    // The next tile: this unit's next, or the first tile of the block's next
    // unit, so the copies run ahead across planes and segments too.
    int64_t nunit = unit, ni = i + 1;
    if (ni >= cu.tiles) {
      nunit = unit + gridDim.x;
      ni = 0;
    }
    const bool more = nunit < units;
    const Unit nu = (more && nunit != unit) ? unit_at(nunit) : cu;
    float* buf = s_dyn + cur * kCap;
    if (more) {
      __syncthreads();  // the other buffer's last tile has been stored
      issue(s_dyn + (cur ^ 1) * kCap, nu, ni, Gt, St, It);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // tile i is in shared memory for every thread
    // Scan this thread's U rows (scan order u = 0 .. U-1).
    float* base_p = buf + (p.reverse ? (Gt - 1 - g) : g) * St + col;
    float q[U][VEC];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float* src = base_p + (p.reverse ? (U - 1 - u) : u) * It;
      if constexpr (VEC == 4) {
        const float4 f = active ? *reinterpret_cast<const float4*>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
        q[u][0] = f.x;
        q[u][1] = f.y;
        q[u][2] = f.z;
        q[u][3] = f.w;
      } else {
        q[u][0] = active ? src[0] : 0.f;
      }
    }
#pragma unroll
    for (int u = 1; u < U; ++u)
#pragma unroll
      for (int c = 0; c < VEC; ++c) q[u][c] += q[u - 1][c];
    float tot[VEC], pre[VEC], b[VEC];
    if (wide_groups) {
      // Row groups of whole warps: their totals through shared memory.
#pragma unroll
      for (int c = 0; c < VEC; ++c) s_tot[g * gcols + col + c] = q[U - 1][c];
      __syncthreads();
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        float r = 0.f, gp = 0.f;
        for (int g2 = 0; g2 < Gt; ++g2) {
          if (g2 == g) gp = r;
          r += s_tot[g2 * gcols + col + c];
        }
        tot[c] = r;
        pre[c] = gp;
      }
    } else {
      // Row groups of this warp: inclusive shuffle scan over them (stride
      // tpr lanes), the exclusive value from the group before, and the warp
      // totals in a fixed order.
      float ex[VEC];
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        float v = q[U - 1][c];
        for (int d = tpr; d < 32; d <<= 1) {
          const float w = __shfl_up_sync(kFullMask, v, d);
          if (lane >= d) v += w;
        }
        const float e = __shfl_up_sync(kFullMask, v, tpr);
        ex[c] = lane >= tpr ? e : 0.f;
        const float wt = __shfl_sync(kFullMask, v, (gpw - 1) * tpr + cg);
        if (lane < tpr) s_tot[warp * 32 * VEC + col + c] = wt;
      }
      __syncthreads();
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        float r = 0.f, wp = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kNW; ++w2) {
          if (w2 == warp) wp = r;
          r += s_tot[w2 * 32 * VEC + col + c];
        }
        tot[c] = r;
        pre[c] = wp + ex[c];
      }
    }
#pragma unroll
    for (int c = 0; c < VEC; ++c) b[c] = tc.base(c);
    // Results back to this thread's places in the tile.
    if (active) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float out[VEC];
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
          const float own = p.exclusive ? (u > 0 ? q[u - 1][c] : 0.f) : q[u][c];
          out[c] = b[c] + (pre[c] + own);
        }
        float* dst = base_p + (p.reverse ? (U - 1 - u) : u) * It;
        if constexpr (VEC == 4)
          *reinterpret_cast<float4*>(dst) = make_float4(out[0], out[1], out[2], out[3]);
        else
          dst[0] = out[0];
      }
    }
    __syncthreads();
    // Store the tile (contiguous), the mapping of the copy in.
    if (active) {
      const int64_t pl = phys_lo(cu, i);
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int pr = k * Gt + g;
        const int64_t row = pl + pr;
        if (row >= cu.lo && row < cu.lo + cu.len) {
          const float* src = buf + (pr / U) * St + (pr % U) * It + col;
          float v[VEC];
          if constexpr (VEC == 4) {
            const float4 f = *reinterpret_cast<const float4*>(src);
            v[0] = f.x;
            v[1] = f.y;
            v[2] = f.z;
            v[3] = f.w;
          } else {
            v[0] = src[0];
          }
          store_vec<VEC>(cu.yo + row * inner, v);
        }
      }
    }
    tc.add(tot);
    cur ^= 1;
    if (!more) break;
    if (nunit != unit) {
      unit = nunit;
      cu = nu;
      tc = carry_of(unit);
    }
    i = ni;
  }
}

// ---------------------------------------------------------------------------
// Warp forms: one warp per (o, segment), no barriers and no shared memory.
// Lane (g, cg): g < Gw = 32 / tpr row groups, cg < tpr column groups; step k
// covers Gw consecutive rows (scan order k*Gw + g), one contiguous load.
//  * scan: U steps loaded at once; each step is scanned over g with shuffles
//    (stride tpr lanes), output = base + (that inclusive or exclusive value),
//    base the blocked running sum of the earlier steps' totals;
//  * reduction: blocked accumulators over the steps, then a shuffle tree over g.
// ---------------------------------------------------------------------------
template <int VEC, int U>
__global__ void __launch_bounds__(kThreads) k_scan_narrow_warp(ScanColsParams p) {
  pdl_begin();
  const int64_t inner = p.inner;
  int tpr = 1;
  while (tpr * VEC < inner) tpr <<= 1;
  const int gw = 32 / tpr;
  const int lane = threadIdx.x & 31;
  const int g = lane / tpr;
  const int cg = lane - g * tpr;
  const int col = cg * VEC;
  const bool active = col < inner;  // with VEC == 4, inner % 4 == 0: all four columns
  const int64_t units = p.outer * p.segs;
  const int64_t wstride = (int64_t)gridDim.x * kNW;
  for (int64_t unit = (int64_t)blockIdx.x * kNW + (threadIdx.x >> 5); unit < units; unit += wstride) {
    const int64_t o = unit / p.segs;
    const int64_t lo = (unit - o * p.segs) * p.seg_len;
    const int64_t len = min(p.seg_len, p.N - lo);
    // Scan-order row s is physical row j0 + s*dir.
    const int64_t j0 = p.reverse ? lo + len - 1 : lo;
    const int64_t dir = p.reverse ? -1 : 1;
    const int64_t off = (o * p.N + j0) * inner + (active ? col : 0);
    const float* xp = p.x + off;
    float* yp = p.y + off;
    float init[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c)
      init[c] = (p.carry != nullptr && active) ? ld_plain(p.carry + unit * p.carry_stride + col + c) : 0.f;
    TileCarry<VEC> tc(init);
    for (int64_t s0 = 0; s0 < len; s0 += (int64_t)U * gw) {
      int64_t step = dir * inner;  // hidden from the optimiser: see k_scan_cols
      asm volatile("" : "+l"(step));
      float q[U][VEC];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t srow = s0 + (int64_t)u * gw + g;
        if (active && srow < len) {
          load_vec<VEC>(q[u], xp + srow * step);
        } else {
#pragma unroll
          for (int c = 0; c < VEC; ++c) q[u][c] = 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float out[VEC];
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
          float v = q[u][c];
          for (int d = tpr; d < 32; d <<= 1) {
            const float w = __shfl_up_sync(kFullMask, v, d);
            if (lane >= d) v += w;
          }
          const float e = __shfl_up_sync(kFullMask, v, tpr);
          const float own = p.exclusive ? (lane >= tpr ? e : 0.f) : v;
          out[c] = tc.base(c) + own;
          q[u][c] = __shfl_sync(kFullMask, v, (gw - 1) * tpr + cg);  // the step's total
        }
        const int64_t srow = s0 + (int64_t)u * gw + g;
        if (active && srow < len) store_vec<VEC>(yp + srow * step, out);
        tc.add(q[u]);
      }
    }
  }
}

template <int VEC, int U, typename Op>
__global__ void __launch_bounds__(kThreads) k_reduce_narrow_warp(NarrowParams p) {
  pdl_begin();
  const int64_t inner = p.inner;
  const int tpr = (int)(inner / VEC);  // <= 32; inner % VEC == 0
  const int gw = 32 / tpr;
  const int lane = threadIdx.x & 31;
  const int g = lane / tpr;
  const int cg = lane - g * tpr;
  const bool active = g < gw;
  const int64_t o = (int64_t)blockIdx.x * kNW + (threadIdx.x >> 5);
  if (o >= p.outer) return;
  float res[VEC];
#pragma unroll
  for (int c = 0; c < VEC; ++c) res[c] = Op::identity();
  if (active) {
    const float* xc = p.x + o * p.reduce * inner + cg * VEC;
    BlockedAcc<kFold, Op> acc[VEC];
    int64_t r = g;
    for (; r + (int64_t)(U - 1) * gw < p.reduce; r += (int64_t)U * gw) {
      float q[U][VEC];
#pragma unroll
      for (int u = 0; u < U; ++u) load_vec<VEC>(q[u], xc + (r + (int64_t)u * gw) * inner);
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        float e[U];
#pragma unroll
        for (int u = 0; u < U; ++u) e[u] = Op::prep(q[u][c]);
        acc[c].add(tree_reduce<Op, U>(e));
      }
    }
    for (; r < p.reduce; r += gw) {
      float q[VEC];
      load_vec<VEC>(q, xc + r * inner);
#pragma unroll
      for (int c = 0; c < VEC; ++c) acc[c].add(Op::prep(q[c]));
    }
#pragma unroll
    for (int c = 0; c < VEC; ++c) res[c] = acc[c].total();
  }
  // Fixed tree over the row groups: lane l takes lane l + d (same column group).
  int gp = 1;
  while (gp < gw) gp <<= 1;
  for (int d = (gp >> 1) * tpr; d >= tpr; d >>= 1) {
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
      const float w = __shfl_down_sync(kFullMask, res[c], d);
      if (lane + d < gw * tpr) res[c] = Op::combine(res[c], w);
    }
  }
  if (g == 0) {
#pragma unroll
    for (int c = 0; c < VEC; ++c) st_plain(p.out + o * inner + cg * VEC + c, finish(res[c], p.epi, p.reduce));
  }
}

}  // namespace

cudaError_t launch_scan_narrow_warp(int vec, const ScanColsParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  if (vec == 4) launch_pdl(k_scan_narrow_warp<4, 8>, g, kThreads, 0, s, p);
  else launch_pdl(k_scan_narrow_warp<1, 8>, g, kThreads, 0, s, p);
  return cudaGetLastError();
}

int occupancy_scan_narrow_warp(int vec) {
  return vec == 4 ? occupancy_of(k_scan_narrow_warp<4, 8>) : occupancy_of(k_scan_narrow_warp<1, 8>);
}

cudaError_t launch_reduce_narrow_warp(int vec, int op, const NarrowParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  constexpr int U = 8;
#define LR_NARROW_WARP_CASE(V, OP)                                 \
  if (vec == V && op == k##OP) {                                   \
    launch_pdl(k_reduce_narrow_warp<V, U, OP>, g, kThreads, 0, s, p);      \
    return cudaGetLastError();                                     \
  }
  LR_NARROW_WARP_CASE(1, OpSum)
  LR_NARROW_WARP_CASE(1, OpSumSq)
  LR_NARROW_WARP_CASE(1, OpMax)
  LR_NARROW_WARP_CASE(1, OpMin)
  LR_NARROW_WARP_CASE(4, OpSum)
  LR_NARROW_WARP_CASE(4, OpSumSq)
  LR_NARROW_WARP_CASE(4, OpMax)
  LR_NARROW_WARP_CASE(4, OpMin)
#undef LR_NARROW_WARP_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_reduce_narrow(int vec, int op, const NarrowParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  constexpr int U = 8;
#define LR_NARROW_CASE(V, OP)                                      \
  if (vec == V && op == k##OP) {                                   \
    launch_pdl(k_reduce_narrow<V, U, OP>, g, kThreads, 0, s, p);           \
    return cudaGetLastError();                                     \
  }
  LR_NARROW_CASE(1, OpSum)
  LR_NARROW_CASE(1, OpSumSq)
  LR_NARROW_CASE(1, OpMax)
  LR_NARROW_CASE(1, OpMin)
  LR_NARROW_CASE(4, OpSum)
  LR_NARROW_CASE(4, OpSumSq)
  LR_NARROW_CASE(4, OpMax)
  LR_NARROW_CASE(4, OpMin)
#undef LR_NARROW_CASE
  return cudaErrorInvalidValue;
}

int occupancy_reduce_narrow(int vec, int op) {
  constexpr int U = 8;
  switch (op) {
    case kOpSum: return vec == 4 ? occupancy_of(k_reduce_narrow<4, U, OpSum>) : occupancy_of(k_reduce_narrow<1, U, OpSum>);
    case kOpSumSq: return vec == 4 ? occupancy_of(k_reduce_narrow<4, U, OpSumSq>) : occupancy_of(k_reduce_narrow<1, U, OpSumSq>);
    case kOpMax: return vec == 4 ? occupancy_of(k_reduce_narrow<4, U, OpMax>) : occupancy_of(k_reduce_narrow<1, U, OpMax>);
    case kOpMin: return vec == 4 ? occupancy_of(k_reduce_narrow<4, U, OpMin>) : occupancy_of(k_reduce_narrow<1, U, OpMin>);
    default: return 0;
  }
}

// The block-form scan keeps two tile buffers in dynamic shared memory (above
// the 48 KiB a launch gets without asking).
template <int VEC, int U>
cudaError_t scan_narrow_kernel(void (**k)(ScanColsParams), size_t* bytes) {
  *k = k_scan_narrow<VEC, U>;
  *bytes = 2 * sizeof(float) * scan_narrow_cap<VEC, U>();
  return cudaFuncSetAttribute(*k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)*bytes);
}

cudaError_t launch_scan_narrow(int vec, const ScanColsParams& p, int64_t grid, cudaStream_t s) {
  void (*k)(ScanColsParams) = nullptr;
  size_t bytes = 0;
  const cudaError_t e = vec == 4 ? scan_narrow_kernel<4, 8>(&k, &bytes) : scan_narrow_kernel<1, 16>(&k, &bytes);
  if (e != cudaSuccess) return e;
  launch_pdl(k, dim3((unsigned)grid), kThreads, bytes, s, p);
  return cudaGetLastError();
}

int occupancy_scan_narrow(int vec) {
  void (*k)(ScanColsParams) = nullptr;
  size_t bytes = 0;
  if ((vec == 4 ? scan_narrow_kernel<4, 8>(&k, &bytes) : scan_narrow_kernel<1, 16>(&k, &bytes)) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, bytes) != cudaSuccess) return 0;
  return n;
}

int64_t scan_narrow_tile_rows(int vec, int64_t inner) {
  int tpr = 1;
  while (tpr * vec < inner) tpr <<= 1;
  return (int64_t)(kThreads / tpr) * (vec == 4 ? 8 : 16);
}

}  // namespace lr
