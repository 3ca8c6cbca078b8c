// lr_scan_cols_lb.cu -- cumulative sum along a strided axis in one pass: a
// decoupled look-back over column tiles, for shapes whose (o, column tile)
// units are too few to fill the GPU one block per unit.
//
// x and y are [outer, N, inner], scanned along N.  The axis of every unit
// (o, 32-column tile) is cut into tiles of 256 rows.  Block t (tickets in
// order, column tile fastest, so the blocks in flight cover whole rows):
//   1. copies tile t into shared memory, in flight meanwhile (float4 rows:
//      one tensor copy by the TMA engine, issued as soon as the ticket is
//      known; other rows: cp.async by every thread),
//   2. rereads tile t - lag into registers (from L2: its first touch was
//      `lag` tickets earlier),
//   3. computes that tile's carry: the tiles before tile k of its unit are,
//      for every level L, the siblings that precede k's level-L ancestor in a
//      32-ary grouping, so each column's carry is the sum over levels (the
//      lowest first) of a fixed-tree sum of at most 31 published words,
//   4. scans it -- a sequential prefix over each thread's rows, the row
//      groups and warps before it in a fixed order, plus the carry -- and
//      writes it,
//   5. sums tile t's columns, publishes them, and publishes every group sum
//      that tile t completes (it is the last child of that group).
// Node words are {epoch:32, fp32:32}, one per column, written and read with
// relaxed single-copy-atomic accesses as in the row look-back; tickets and
// the launch epoch come from the same 64-bit word.  Every sum runs in a
// fixed order, so reruns are bit-identical, and no output subtracts anything.
// Forward progress: a tile waits only on tiles of its own unit with smaller
// k, hence smaller tickets; every wait is bounded.
#include <cuda.h>  // CUtensorMap

#include <cstring>

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

constexpr int kNW = kColLbWarps;
constexpr int kLbThreads = 32 * kNW;
constexpr int TR = kColLbRows;
constexpr int kColsPerWarp = kColLbCols / kNW;  // publication: warp w owns these columns
constexpr int kSibPerWarp = (31 + kNW - 1) / kNW;  // look-back siblings a warp reads per level
static_assert(kColLbCols == 32 && kColLbCols % kNW == 0, "a 32-column tile, whole columns per warp");
constexpr int kRowsPerWarp = TR / kNW;  // a warp covers this many consecutive rows of a tile
static_assert(kRowsPerWarp == 32, "every thread owns whole rows");
constexpr int kBoxRows = 256;  // a tensor copy moves at most 256 rows
static_assert(TR % kBoxRows == 0, "whole boxes per tile");

struct TilePos {
  int o, k, ct;  // tickets and tile counts fit 31 bits (the host caps the tiles of a launch)
};

// Tickets and tile counts fit 32 bits (the host caps the tiles of a launch),
// so the divisions are 32-bit; one thread computes them for the block.
__device__ __forceinline__ TilePos tile_pos(int ticket, int tiles, int col_tiles) {
  const unsigned tk = (unsigned)ticket, per_o = (unsigned)tiles * (unsigned)col_tiles, ct = (unsigned)col_tiles;
  const unsigned o = tk / per_o;
  const unsigned r = tk - o * per_o;
  const unsigned k = r / ct;
  return TilePos{(int)o, (int)k, (int)(r - k * ct)};
}

// Offset in x and y of scan position n (< N) of column col of outer index o.
__device__ __forceinline__ int64_t elem_off(const ScanColsLookbackParams& p, int64_t o, int64_t n,
                                            int64_t col) {
  return (o * p.N + (p.reverse ? p.N - 1 - n : n)) * p.inner + col;
}

__device__ __forceinline__ unsigned long long* unit_nodes(const ScanColsLookbackParams& p, const TilePos& q) {
  return p.node_val + ((int64_t)q.o * p.col_tiles + q.ct) * 2 * p.tiles * kColLbCols;
}

// Thread layout of a TR x 32 tile with VEC-wide items: LPR = 32 / VEC lanes
// across a row, RG = VEC row groups per warp, R = kRowsPerWarp / VEC
// consecutive rows (in scan order) per thread.  Thread (w, lane) owns columns
// cg*VEC .. cg*VEC + VEC-1 (cg = lane % LPR) of rows w*kRowsPerWarp + rq*R ..
// + R-1 (rq = lane / LPR); it copies, sums, rereads, scans and writes exactly
// those.
template <int VEC>
struct Layout {
  static constexpr int LPR = 32 / VEC;
  static constexpr int RG = VEC;
  static constexpr int R = kRowsPerWarp / VEC;
};

// Pointer to the thread's first element of tile q (scan position
// k*256 + w*32 + rq*R) and the number of its rows inside the axis.
template <int VEC>
__device__ __forceinline__ const float* tile_ptr(const ScanColsLookbackParams& p, const float* base,
                                                 const TilePos& q, int w, int lane, int* rows, bool* cok) {
  using Ly = Layout<VEC>;
  const int64_t col = (int64_t)q.ct * kColLbCols + (lane % Ly::LPR) * VEC;
  const int64_t n0 = (int64_t)q.k * TR + w * kRowsPerWarp + (lane / Ly::LPR) * Ly::R;
  *rows = (int)max((int64_t)0, min((int64_t)Ly::R, p.N - n0));
  *cok = col < p.inner;  // with VEC 4, inner % 4 == 0: all four columns or none
  return (*rows > 0 && *cok) ? base + elem_off(p, q.o, n0, col) : base;
}

template <int VEC>
__device__ __forceinline__ void load_item(float (&d)[VEC], const float* src) {
  if constexpr (VEC == 4) {
    const float4 f = ld_stream4(src);
    d[0] = f.x;
    d[1] = f.y;
    d[2] = f.z;
    d[3] = f.w;
  } else {
    d[0] = ld_stream1(src);
  }
}

// The node words of one lane (columns col0 .. col0+kColsPerWarp-1 of one node):
// read them, then poll the ones that do not yet carry this launch's epoch
// until they do (bounded: on giving up *fail is set and they read as 0).
__device__ __forceinline__ void read_words(const unsigned long long* src, bool active, unsigned epoch,
                                           const ScanColsLookbackParams& p, const unsigned* abort_word,
                                           float (&out)[kColsPerWarp], bool* fail) {
  unsigned long long word[kColsPerWarp];
#pragma unroll
  for (int c = 0; c < kColsPerWarp; ++c) word[c] = active ? ld_relaxed_u64(src + c) : 0ull;
  const auto ready = [&]() {
    bool r = true;
#pragma unroll
    for (int c = 0; c < kColsPerWarp; ++c) r = r && (unsigned)(word[c] >> 32) == epoch;
    return r;
  };
  if (active && !ready()) {
    unsigned ns = 0;
    for (int64_t it = 0; !ready(); ++it) {
      if (it >= p.spin_limit || ld_relaxed_u32(abort_word) == epoch) {
        *fail = true;
        break;
      }
      if (it >= 64) {  // spin first, then back off gently
        ns = ns ? (ns < 256 ? 2 * ns : ns) : 32;
        __nanosleep(ns);
      }
#pragma unroll
      for (int c = 0; c < kColsPerWarp; ++c)
        if ((unsigned)(word[c] >> 32) != epoch) word[c] = ld_relaxed_u64(src + c);
    }
  }
#pragma unroll
  for (int c = 0; c < kColsPerWarp; ++c)
    out[c] = (active && (unsigned)(word[c] >> 32) == epoch) ? __uint_as_float((unsigned)word[c]) : 0.f;
}

__device__ __forceinline__ float pick(const float (&a)[kColsPerWarp], int i) {
  float r = a[0];
#pragma unroll
  for (int c = 1; c < kColsPerWarp; ++c)
    if (i == c) r = a[c];
  return r;
}

// VEC 4 (inner % 4 == 0, x and y 16-byte aligned) copies tiles with the
// tensor map `tmap` ([outer, N, inner] fp32, box 32 x 256 x 1); VEC 1 ignores it.
// The tile lands in dynamic shared memory (TR x 32 floats).
template <int VEC>
__global__ void __launch_bounds__(kLbThreads, 32 / kNW) k_scan_cols_lookback(
    ScanColsLookbackParams p, const __grid_constant__ CUtensorMap tmap) {
  pdl_begin();
  using Ly = Layout<VEC>;
  constexpr int R = Ly::R;
  constexpr bool kTma = VEC == 4;
  extern __shared__ __align__(128) float s_tile_mem[];
  float(*s_tile)[kColLbCols] = reinterpret_cast<float(*)[kColLbCols]>(s_tile_mem);
  __shared__ unsigned long long s_bar;
  __shared__ __align__(16) float s_tot[kNW][kColLbCols];  // warp totals of the reread tile
  __shared__ __align__(16) float s_sum[kNW][kColLbCols];  // warp sums of the copied tile
  __shared__ __align__(16) float s_part[kColLbMaxLevels][kNW][kColLbCols];  // look-back partials per warp
  __shared__ unsigned s_ticket, s_epoch;
  __shared__ TilePos s_pos[2];  // tile `ticket` and tile `ticket - lag`
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int w = t >> 5;
  const int cg = lane % Ly::LPR;
  const int rq = lane / Ly::LPR;
  const unsigned* abort_word = p.err_word + 1;
  const int K = (int)p.tiles;
  const int CT = (int)p.col_tiles;
  const int lag = (int)p.lag;
  const int total = (int)(p.outer * p.tiles * p.col_tiles);

  if (t == 0) {
    const Ticket tkt = take_ticket(p.ticket_word);
    s_ticket = tkt.ticket;
    s_epoch = tkt.epoch;
    // Every other ticket is taken before the last one: reset for the next launch.
    if ((int64_t)tkt.ticket == (int64_t)total + lag - 1) next_launch(p.ticket_word, tkt.epoch);
    const int tk = (int)tkt.ticket;
    const TilePos q = tk < total ? tile_pos(tk, K, CT) : TilePos{0, 0, 0};
    s_pos[0] = q;
    s_pos[1] = (tk >= lag && tk - lag < total) ? tile_pos(tk - lag, K, CT) : TilePos{0, 0, 0};
    if (kTma && tk < total) {
      // The tile's first row in memory: scan positions k*TR .. k*TR+TR-1 are
      // rows N-1-k*TR down to N-TR-k*TR when reverse (possibly negative).
      const int64_t row0 = p.reverse ? p.N - (int64_t)(q.k + 1) * TR : (int64_t)q.k * TR;
      mbar_init(&s_bar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&s_bar, (unsigned)(TR * kColLbCols * sizeof(float)));
#pragma unroll
      for (int b = 0; b < TR / kBoxRows; ++b)
        tma_load_3d(&s_tile[b * kBoxRows][0], &tmap, (int)(q.ct * kColLbCols), (int)(row0 + b * kBoxRows),
                    (int)q.o, &s_bar);
    }
  }
  __syncthreads();
  const unsigned epoch = s_epoch;
  if ((int64_t)s_ticket >= (int64_t)total + lag) {  // a stale counter: touch nothing
    if (t == 0) atomicOr(p.err_word, 2u);
    return;
  }
  const int ticket = (int)s_ticket;
  const int64_t step = p.reverse ? -p.inner : p.inner;  // from one scan position to the next
  int levels = 1;
  while (levels < kColLbMaxLevels && ((K - 1) >> (5 * levels)) != 0) ++levels;
  float* my_tile = &s_tile[w * kRowsPerWarp + rq * R][cg * VEC];  // row i of mine: my_tile + i * 32
  const int col0 = w * kColsPerWarp;                    // this warp's look-back columns
  bool fail = false;

  // ---- 1. copy my part of tile `ticket` into shared memory (VEC 1) ----
  int rows_t = 0;
  bool cok_t = false;
  if (!kTma && ticket < total) {
    const float* src = tile_ptr<VEC>(p, p.x, s_pos[0], w, lane, &rows_t, &cok_t);
    if (cok_t) {
#pragma unroll
      for (int i = 0; i < R; ++i) {
        if (i < rows_t) {
          cp_async4(my_tile + i * 32, src, 4u);
          src += step;
        }
      }
    }
    cp_async_commit();
  }

  // ---- 2. reread tile u = ticket - lag (from L2) ----
  const int u = ticket - lag;
  float v[R][VEC];
  int rows_u = 0;
  bool cok_u = false;
  if (u >= 0) {
    const float* src = tile_ptr<VEC>(p, p.x, s_pos[1], w, lane, &rows_u, &cok_u);
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (cok_u && i < rows_u) {
        load_item<VEC>(v[i], src);
        src += step;
      } else {
#pragma unroll
        for (int c = 0; c < VEC; ++c) v[i][c] = 0.f;
      }
    }

    // ---- 3. look-back of tile u: warp w reads siblings w, w+8, w+16, w+24
    // of every level, lane = column (one 256-byte node row per load), and
    // leaves its per-level partial sums (siblings in order) in s_part ----
    const TilePos qu = s_pos[1];
    const unsigned long long* vals = unit_nodes(p, qu);
    int off = 0, count = K;
    for (int L = 0; L < levels; ++L) {
      const int m = qu.k >> (5 * L);
      const int d = (int)(m & 31);
      const unsigned long long* sib = vals + (off + m - d) * kColLbCols + lane;
      unsigned long long word[kSibPerWarp];
#pragma unroll
      for (int i = 0; i < kSibPerWarp; ++i)
        word[i] = w + kNW * i < d ? ld_relaxed_u64(sib + (w + kNW * i) * kColLbCols) : 0ull;
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < kSibPerWarp; ++i) {
        if (w + kNW * i < d)
          part += (unsigned)(word[i] >> 32) == epoch
                      ? __uint_as_float((unsigned)word[i])
                      : wait_node(sib + (w + kNW * i) * kColLbCols, epoch, p.spin_limit, abort_word, &fail);
      }
      s_part[L][w][lane] = part;
      off += count;
      count >>= 5;
    }
  } else {
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int c = 0; c < VEC; ++c) v[i][c] = 0.f;
  }

  // ---- 4. scan tile u and write it ----
  // Sequential prefix over my R rows, to which the row groups before mine in
  // this warp are added before the barrier; after it the carry and the warps
  // before mine (fixed orders).
#pragma unroll
  for (int c = 0; c < VEC; ++c) {
    float run = 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const float before = run;
      run += v[i][c];
      v[i][c] = p.exclusive ? before : run;
    }
    float acc = 0.f, wt = 0.f;
#pragma unroll
    for (int g = 0; g < Ly::RG; ++g) {
      const float tg = Ly::RG > 1 ? __shfl_sync(kFullMask, run, g * Ly::LPR + cg) : run;
      if (g < rq) acc += tg;
      wt += tg;
    }
#pragma unroll
    for (int i = 0; i < R; ++i) v[i][c] = acc + v[i][c];
    if (rq == 0) s_tot[w][cg * VEC + c] = wt;  // the warp's column totals
  }
  __syncthreads();  // s_tot and s_part complete
  if (u >= 0 && cok_u) {
    // carry = sum over levels (lowest first) of the warp partials in warp
    // order; base = carry + warps before mine.
    float carry[VEC], wsum[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) carry[c] = wsum[c] = 0.f;
    for (int L = 0; L < levels; ++L) {
      float lv[VEC];
#pragma unroll
      for (int c = 0; c < VEC; ++c) lv[c] = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kNW; ++w2) {
        if constexpr (VEC == 4) {
          const float4 q = *reinterpret_cast<const float4*>(&s_part[L][w2][cg * 4]);
          lv[0] += q.x;
          lv[1] += q.y;
          lv[2] += q.z;
          lv[3] += q.w;
        } else {
          lv[0] += s_part[L][w2][cg];
        }
      }
#pragma unroll
      for (int c = 0; c < VEC; ++c) carry[c] += lv[c];
    }
    for (int w2 = 0; w2 < w; ++w2) {
      if constexpr (VEC == 4) {
        const float4 q = *reinterpret_cast<const float4*>(&s_tot[w2][cg * 4]);
        wsum[0] += q.x;
        wsum[1] += q.y;
        wsum[2] += q.z;
        wsum[3] += q.w;
      } else {
        wsum[0] += s_tot[w2][cg];
      }
    }
    float basev[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) basev[c] = carry[c] + wsum[c];
    // The stride is hidden from the optimiser here: otherwise it reuses the
    // row addresses of the reread and holds them all in registers.
    int64_t st = step;
    asm volatile("" : "+l"(st));
    float* dst = const_cast<float*>(tile_ptr<VEC>(p, p.y, s_pos[1], w, lane, &rows_u, &cok_u));
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (i < rows_u) {
        if constexpr (VEC == 4)
          st_stream4(dst, make_float4(basev[0] + v[i][0], basev[1] + v[i][1], basev[2] + v[i][2],
                                      basev[3] + v[i][3]));
        else
          st_stream1(dst, basev[0] + v[i][0]);
        dst += st;
      }
    }
  }

  // ---- 5. sum tile `ticket`, publish it and the group sums it completes ----
  if (ticket < total) {
    if constexpr (kTma) {
      // The whole box, zeros outside the tensor: every thread sums its rows.
      // The copy is waited for with a time bound independent of the poll
      // limit, so the block never leaves while it is in flight.
      if (!mbar_wait_copy(&s_bar, 0u)) fail = true;
      rows_t = R;
      cok_t = true;
    } else {
      cp_async_wait<0>();  // my own copies: no barrier needed to read them
    }
    // Whole items (a float4 per row) keep the shared-memory reads free of
    // bank conflicts.
    float a[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) a[c] = 0.f;
    if (cok_t) {
#pragma unroll
      for (int i = 0; i < R; ++i) {
        if (i < rows_t) {
          if constexpr (VEC == 4) {
            const float4 q = *reinterpret_cast<const float4*>(my_tile + i * 32);
            a[0] += q.x;
            a[1] += q.y;
            a[2] += q.z;
            a[3] += q.w;
          } else {
            a[0] += my_tile[i * 32];
          }
        }
      }
    }
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
      float ws = 0.f;
#pragma unroll
      for (int g = 0; g < Ly::RG; ++g) ws += Ly::RG > 1 ? __shfl_sync(kFullMask, a[c], g * Ly::LPR + cg) : a[c];
      if (rq == 0) s_sum[w][cg * VEC + c] = ws;
    }
    __syncthreads();
    // Warp w publishes columns col0 .. col0+3: the tile's sums (warps in
    // order), then each group sum the tile completes (a fixed tree over the
    // 32 children, the tile's own ancestor in lane 31).
    const TilePos q = s_pos[0];
    unsigned long long* vals = unit_nodes(p, q);
    const bool stalled = ticket == p.stall_tile;
    float own[kColsPerWarp];
#pragma unroll
    for (int c = 0; c < kColsPerWarp; ++c) {
      float a = 0.f;
      for (int w2 = 0; w2 < kNW; ++w2) a += s_sum[w2][col0 + c];
      own[c] = a;
    }
    if (!stalled) {
      if (lane < kColsPerWarp)
        st_relaxed_u64(vals + q.k * kColLbCols + col0 + lane, pack_node(epoch, pick(own, lane)));
      int off = 0, count = K, m = q.k;
      for (int L = 0; L + 1 < levels && (m & 31) == 31; ++L) {
        float val[kColsPerWarp];
        bool f2 = false;
        read_words(vals + (off + m - 31 + lane) * kColLbCols + col0, lane < 31, epoch, p, abort_word, val, &f2);
#pragma unroll
        for (int c = 0; c < kColsPerWarp; ++c)
          own[c] = __shfl_sync(kFullMask, warp_tree_adjacent(lane < 31 ? val[c] : own[c]), 0);
        if (__any_sync(kFullMask, f2)) {
          fail = true;
          break;
        }
        const int next_off = off + count;
        if (lane < kColsPerWarp)
          st_relaxed_u64(vals + (next_off + (m >> 5)) * kColLbCols + col0 + lane, pack_node(epoch, pick(own, lane)));
        off = next_off;
        count >>= 5;
        m >>= 5;
      }
    }
  }
  if (__any_sync(kFullMask, fail) && lane == 0) {
    atomicOr(p.err_word, 1u);
    atomicExch(p.err_word + 1, epoch);
  }
}

}  // namespace

// The tensor-map encoder, from the driver through the runtime (no link
// against the driver library); null where unavailable.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Tensor map of x as [outer, N, inner] fp32 with a box of 32 columns x 256
// rows x 1 plane.  Needs inner % 4 == 0 and x 16-byte aligned (the strides
// and the base must be multiples of 16 bytes).
bool encode_cols_map(CUtensorMap* m, const ScanColsLookbackParams& p) {
  const EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr || p.inner % 4 != 0 || (reinterpret_cast<uintptr_t>(p.x) & 15u) != 0 || p.N >= INT32_MAX ||
      p.outer >= INT32_MAX || p.inner >= INT32_MAX)
    return false;
  const cuuint64_t dims[3] = {(cuuint64_t)p.inner, (cuuint64_t)p.N, (cuuint64_t)p.outer};
  const cuuint64_t strides[2] = {(cuuint64_t)p.inner * 4, (cuuint64_t)p.N * (cuuint64_t)p.inner * 4};
  const cuuint32_t box[3] = {kColLbCols, kBoxRows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(p.x), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t kTileBytes = (size_t)TR * kColLbCols * sizeof(float);  // dynamic shared memory

cudaError_t launch_scan_cols_lookback(int vec, const ScanColsLookbackParams& p, int64_t grid, cudaStream_t s) {
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  if (vec == 4 && encode_cols_map(&m, p))
    launch_pdl(k_scan_cols_lookback<4>, dim3((unsigned)grid), kLbThreads, kTileBytes, s, p, m);
  else
    launch_pdl(k_scan_cols_lookback<1>, dim3((unsigned)grid), kLbThreads, kTileBytes, s, p, m);
  return cudaGetLastError();
}

int occupancy_scan_cols_lookback() {
  int n1 = 0, n4 = 0;
  if (cudaFuncSetAttribute(k_scan_cols_lookback<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTileBytes) !=
          cudaSuccess ||
      cudaFuncSetAttribute(k_scan_cols_lookback<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTileBytes) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n1, k_scan_cols_lookback<1>, kLbThreads, kTileBytes) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n4, k_scan_cols_lookback<4>, kLbThreads, kTileBytes) != cudaSuccess)
    return 0;
  return n1 < n4 ? n1 : n4;
}

}  // namespace lr
