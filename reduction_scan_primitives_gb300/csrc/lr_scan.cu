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
#include <algorithm>

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

constexpr int kNW = kThreads / 32;
constexpr int kCarryFold = 32;  // tiles per fold of the blocked carry

// A row as the tile kernels see it.  With float4 items a row of any length
// and any 4-byte alignment is read as a "virtual row" that starts at the
// 16-byte boundary at or before its first element and is padded to a multiple
// of 4: its elements are virtual indices [lo, hi), the rest read as zeros and
// are never written.  Only 16-byte chunks that hold some of the row's
// elements are read, so every read stays inside the row's memory pages.  y
// must share x's 16-byte misalignment (the caller checks).  With scalar items
// the view is the row itself.
struct RowView {
  const float* x;  // virtual index 0 (16-byte aligned for float4 items)
  float* y;
  int64_t V;       // virtual length (a multiple of 4 for float4 items)
  int64_t lo, hi;  // the row's elements
};

// EDGES = false: the caller guarantees whole aligned float4 rows (N % 4 == 0,
// x 16-byte aligned), so the view is the row itself.
template <int VEC, bool EDGES = true>
__device__ __forceinline__ RowView row_view(const float* x, float* y, int64_t row, int64_t N) {
  const float* xr = x + row * N;
  int64_t m = 0;
  if constexpr (VEC == 4 && EDGES) m = (int64_t)((reinterpret_cast<uintptr_t>(xr) >> 2) & 3);
  RowView r;
  r.x = xr - m;
  r.y = y != nullptr ? y + row * N - m : nullptr;
  r.lo = m;
  r.hi = m + N;
  r.V = (VEC == 4 && EDGES) ? ((m + N + 3) & ~(int64_t)3) : N;
  return r;
}

// One tile of a row: virtual elements [base, base + len) of the row, or the
// mirrored ones [V - base - len, V - base) when `mirror` is set (a forward
// scan run as a reverse scan of the mirrored row).  x and y point at the
// tile's lowest element in memory; element jj of the tile (in scan order) is
// x[jj], or x[len - VEC - jj] mirrored, with float4 items' components then
// taken in reverse order.  lo and hi bound the row's own elements relative to
// x.  All tile-relative indices fit 32 bits.
struct TileView {
  const float* x;
  float* y;
  int len, lo, hi;
};

__device__ __forceinline__ TileView tile_view(const RowView& rv, int64_t base, int64_t tile, bool mirror) {
  TileView tv;
  const int64_t len = max((int64_t)0, min(tile, rv.V - base));  // 0: a tile past the row's end
  const int64_t phys = len > 0 ? (mirror ? rv.V - base - len : base) : 0;
  tv.x = rv.x + phys;
  tv.y = rv.y != nullptr ? rv.y + phys : nullptr;
  tv.len = (int)len;
  tv.lo = (int)min(max(rv.lo - phys, (int64_t)0), len);
  tv.hi = (int)min(max(rv.hi - phys, (int64_t)0), len);
  return tv;
}

// Tile loads and stores.  Every float4 item of a virtual row holds at least
// one row element (lo <= 3 and hi > V - 4), so the loads need no edge test: an
// item at the row's edge reads its whole 16-byte granule, which lies in the
// same page as the row element it holds.  The elements outside the row are
// zeroed by mask_tile, called where the tile is consumed: masking right after
// the loads would wait on them and stall a prefetch.  Stores write the row's
// own elements only.
template <int VEC, int SUB>
__device__ __forceinline__ void load_tile(float (&v)[SUB][VEC], const TileView& tv, int t, bool mirror) {
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    const int jj = s * kThreads * VEC + t * VEC;
    if constexpr (VEC == 4) {
      // len % 4 == 0 and jj % 4 == 0, so jj < len means all four are in the tile.
      float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
      if (jj < tv.len) q = ld_stream4(tv.x + (mirror ? tv.len - 4 - jj : jj));
      if (mirror) {
        v[s][0] = q.w;
        v[s][1] = q.z;
        v[s][2] = q.y;
        v[s][3] = q.x;
      } else {
        v[s][0] = q.x;
        v[s][1] = q.y;
        v[s][2] = q.z;
        v[s][3] = q.w;
      }
    } else {
      v[s][0] = (jj < tv.len) ? ld_stream1(tv.x + (mirror ? tv.len - 1 - jj : jj)) : 0.f;
    }
  }
}

// True when the tile holds an edge of its row (the same in every thread).
__device__ __forceinline__ bool tile_has_edge(const TileView& tv) { return tv.lo > 0 || tv.hi < tv.len; }

// Zeroes the loaded items' components that lie outside the row.
template <int VEC, int SUB>
__device__ __forceinline__ void mask_tile(float (&v)[SUB][VEC], const TileView& tv, int t, bool mirror) {
  if constexpr (VEC == 4) {  // scalar tiles hold row elements only
    if (!tile_has_edge(tv)) return;
#pragma unroll
    for (int s = 0; s < SUB; ++s) {
      const int jj = s * kThreads * 4 + t * 4;
      const int r = mirror ? tv.len - 4 - jj : jj;  // memory offset of the item
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = mirror ? r + 3 - c : r + c;  // memory offset of v[s][c]
        if (e < tv.lo || e >= tv.hi) v[s][c] = 0.f;
      }
    }
  }
}

template <int VEC, int SUB, bool EDGES = true>
__device__ __forceinline__ void store_tile(const float (&v)[SUB][VEC], const TileView& tv, int t, bool mirror) {
  const bool edge = EDGES && VEC == 4 && tile_has_edge(tv);
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    const int jj = s * kThreads * VEC + t * VEC;
    if (jj < tv.len) {
      if constexpr (VEC == 4) {
        const int r = mirror ? tv.len - 4 - jj : jj;
        float q[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) q[c] = mirror ? v[s][3 - c] : v[s][c];
        if (!edge || (r >= tv.lo && r + 4 <= tv.hi)) {
          st_stream4(tv.y + r, make_float4(q[0], q[1], q[2], q[3]));
        } else {  // an edge of the row: its own elements only
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (r + c >= tv.lo && r + c < tv.hi) st_stream1(tv.y + r + c, q[c]);
        }
      } else {
        st_stream1(tv.y + (mirror ? tv.len - 1 - jj : jj), v[s][0]);
      }
    }
  }
}

// Suffix scan of one tile held in registers (v[s][i]: element s*256*VEC +
// t*VEC + i of the tile).  The elements fall into P classes, element e in
// class e % P (P divides VEC, so item component i is in class i % P), and
// each class is scanned on its own: a narrow plane of P columns read as one
// flat row has column c of every row in one class.  P = 1 is the plain row
// scan.  On return v holds each thread's local suffix within each class and
// off[s][c] = exc + (wexc + rs), where exc is the class-c suffix over lanes to
// the right, wexc over warps to the right and rs over sub-tiles to the right
// inside the tile; the caller adds off[s][c] + carry[c] (carry: the tiles to
// the right).  total[c] is the tile's class-c sum (identical in every
// thread).  Contains one __syncthreads(); `sh` must not be written again until
// every thread of the block is past that barrier.
template <int SUB, int P = 1>
struct TileScan {
  float off[SUB][P];
  float total[P];
};

template <int VEC, int SUB, int P = 1>
__device__ __forceinline__ TileScan<SUB, P> tile_suffix(float (&v)[SUB][VEC], float (&sh)[SUB][kNW][P],
                                                       int lane, int w) {
  static_assert(VEC % P == 0, "every item holds whole classes");
  TileScan<SUB, P> r;
  float exc[SUB][P];
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    // 1. Suffix of each thread's VEC items within each class, right to left.
#pragma unroll
    for (int i = VEC - 1 - P; i >= 0; --i) v[s][i] += v[s][i + P];
    // 2. Inclusive suffix over lanes: lane l gets the sum over lanes >= l.
#pragma unroll
    for (int c = 0; c < P; ++c) {
      float a = v[s][c];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_down_sync(kFullMask, a, o);
        if (lane + o < 32) a += u;
      }
      const float e = __shfl_down_sync(kFullMask, a, 1);
      exc[s][c] = (lane == 31) ? 0.f : e;
      if (lane == 0) sh[s][w][c] = a;  // the warp's class-c total
    }
  }
  __syncthreads();
  // 3. Warp totals -> exclusive suffix over warps and sub-tile totals;
  // 4. sub-tiles to the right inside this tile.
  float rs[P];  // sum of the sub-tiles to the right of s
#pragma unroll
  for (int c = 0; c < P; ++c) rs[c] = 0.f;
#pragma unroll
  for (int s = SUB - 1; s >= 0; --s) {
#pragma unroll
    for (int c = 0; c < P; ++c) {
      float wt[kNW];
#pragma unroll
      for (int q = 0; q < kNW; ++q) wt[q] = sh[s][q][c];
      float wexc = 0.f;
#pragma unroll
      for (int q = kNW - 1; q >= 1; --q)
        if (q > w) wexc += wt[q];
      r.off[s][c] = exc[s][c] + (wexc + rs[c]);
      const float stot = tree_sum<kNW>(wt);
      rs[c] = (s == SUB - 1) ? stot : stot + rs[c];
    }
  }
#pragma unroll
  for (int c = 0; c < P; ++c) r.total[c] = rs[c];
  return r;
}

// Turn the local suffixes into outputs: add each sub-tile's offset and the
// carry of the item's class.  Inclusive: item i gets its own local suffix.
// Exclusive: item i gets the local suffix of the next item of its class to
// its right (none for the thread's last item of each class), so no output
// ever subtracts its own term.
template <int VEC, int SUB, int P>
__device__ __forceinline__ void finalize_p(float (&v)[SUB][VEC], const TileScan<SUB, P>& ts,
                                           const float (&carry)[P], bool exclusive) {
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    float off[P];
#pragma unroll
    for (int c = 0; c < P; ++c) off[c] = ts.off[s][c] + carry[c];
    if (exclusive) {
#pragma unroll
      for (int i = 0; i + P < VEC; ++i) v[s][i] = v[s][i + P] + off[i % P];
#pragma unroll
      for (int i = VEC - P; i < VEC; ++i) v[s][i] = off[i % P];
    } else {
#pragma unroll
      for (int i = 0; i < VEC; ++i) v[s][i] += off[i % P];
    }
  }
}
template <int VEC, int SUB>
__device__ __forceinline__ void finalize(float (&v)[SUB][VEC], const TileScan<SUB, 1>& ts, float carry,
                                         bool exclusive) {
  const float c1[1] = {carry};
  finalize_p<VEC, SUB, 1>(v, ts, c1, exclusive);
}

// tile_suffix and finalize_p in one pass, for P > 1 (narrow planes read flat):
// each sub-tile's offsets are applied as soon as they are formed, so no
// SUB x P array of them is held (the same additions in the same order as the
// two calls).  carry_of(c) is evaluated after the barrier, where look-back
// partials published before it are complete.  total[c] gets the tile's
// class sums.
template <int VEC, int SUB, int P, typename CarryFn>
__device__ __forceinline__ void tile_scan_apply(float (&v)[SUB][VEC], float (&sh)[SUB][kNW][P], int lane, int w,
                                                CarryFn carry_of, bool exclusive, float (&total)[P]) {
  static_assert(VEC % P == 0, "every item holds whole classes");
  float exc[SUB][P];
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
#pragma unroll
    for (int i = VEC - 1 - P; i >= 0; --i) v[s][i] += v[s][i + P];
#pragma unroll
    for (int c = 0; c < P; ++c) {
      float a = v[s][c];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_down_sync(kFullMask, a, o);
        if (lane + o < 32) a += u;
      }
      const float e = __shfl_down_sync(kFullMask, a, 1);
      exc[s][c] = (lane == 31) ? 0.f : e;
      if (lane == 0) sh[s][w][c] = a;
    }
  }
  __syncthreads();
  float carry[P], rs[P];
#pragma unroll
  for (int c = 0; c < P; ++c) {
    carry[c] = carry_of(c);
    rs[c] = 0.f;
  }
#pragma unroll
  for (int s = SUB - 1; s >= 0; --s) {
    float off[P];
#pragma unroll
    for (int c = 0; c < P; ++c) {
      float wt[kNW];
#pragma unroll
      for (int q = 0; q < kNW; ++q) wt[q] = sh[s][q][c];
      float wexc = 0.f;
#pragma unroll
      for (int q = kNW - 1; q >= 1; --q)
        if (q > w) wexc += wt[q];
      off[c] = (exc[s][c] + (wexc + rs[c])) + carry[c];
      const float stot = tree_sum<kNW>(wt);
      rs[c] = (s == SUB - 1) ? stot : stot + rs[c];
    }
    if (exclusive) {
#pragma unroll
      for (int i = 0; i + P < VEC; ++i) v[s][i] = v[s][i + P] + off[i % P];
#pragma unroll
      for (int i = VEC - P; i < VEC; ++i) v[s][i] = off[i % P];
    } else {
#pragma unroll
      for (int i = 0; i < VEC; ++i) v[s][i] += off[i % P];
    }
  }
#pragma unroll
  for (int c = 0; c < P; ++c) total[c] = rs[c];
}

// Per-class block sums (fixed trees: warp shuffles, then the warp totals in
// warp 0); the results are valid in warp 0, lane 0.  sh holds kNW x P floats.
template <int P>
__device__ __forceinline__ void block_sum_p(float (&v)[P], float (&sh)[kNW][P]) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
#pragma unroll
  for (int c = 0; c < P; ++c) {
    v[c] = warp_reduce<OpSum>(v[c]);
    if (lane == 0) sh[warp][c] = v[c];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int c = 0; c < P; ++c) {
      float r = lane < kNW ? sh[lane][c] : 0.f;
#pragma unroll
      for (int o = kNW / 2; o > 0; o >>= 1) r += __shfl_down_sync(kFullMask, r, o);
      v[c] = r;
    }
  }
}

// ---------------------------------------------------------------------------
// Block per row: tiles right to left, carry in registers, next tile
// prefetched into registers while the current one is scanned.
// ---------------------------------------------------------------------------
template <int VEC, int SUB, bool EDGES, int P = 1>
__global__ void __launch_bounds__(kThreads) k_rscan_rows(RScanRowsParams p) {
  pdl_begin();
  constexpr int64_t TILE = (int64_t)SUB * kThreads * VEC;
  __shared__ float sh_w[2][SUB][kNW][P];  // warp totals, double-buffered by tile parity
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int w = t >> 5;
  const bool mirror = (p.flags & kScanMirror) != 0;
  const bool exclusive = (p.flags & kScanExclusive) != 0;
  int par = 0;

  for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
    const RowView rv = row_view<VEC, EDGES>(p.x, p.y, row, p.N);
    const int64_t ntiles = (rv.V + TILE - 1) / TILE;
    float cur[SUB][VEC];
    float nxt[SUB][VEC];
    load_tile<VEC, SUB>(cur, tile_view(rv, (ntiles - 1) * TILE, TILE, mirror), t, mirror);
    float carry_lo[P], carry_hi[P];
#pragma unroll
    for (int c = 0; c < P; ++c) carry_lo[c] = carry_hi[c] = 0.f;
    int ncarry = 0;

    for (int64_t k = ntiles - 1; k >= 0; --k) {
      const int64_t base = k * TILE;
      if (k > 0) load_tile<VEC, SUB>(nxt, tile_view(rv, base - TILE, TILE, mirror), t, mirror);  // prefetch
      const TileView tv = tile_view(rv, base, TILE, mirror);
      if constexpr (EDGES) mask_tile<VEC, SUB>(cur, tv, t, mirror);
      float tot[P];
      if constexpr (P == 1) {
        const TileScan<SUB, P> ts = tile_suffix<VEC, SUB, P>(cur, sh_w[par], lane, w);
        finalize<VEC, SUB>(cur, ts, carry_hi[0] + carry_lo[0], exclusive);
        tot[0] = ts.total[0];
      } else {
        tile_scan_apply<VEC, SUB, P>(cur, sh_w[par], lane, w, [&](int c) { return carry_hi[c] + carry_lo[c]; },
                                     exclusive, tot);
      }
      store_tile<VEC, SUB, EDGES>(cur, tv, t, mirror);
      // Blocked carry: fold every kCarryFold tiles to keep chains short.
#pragma unroll
      for (int c = 0; c < P; ++c) carry_lo[c] += tot[c];
      if (++ncarry == kCarryFold) {
#pragma unroll
        for (int c = 0; c < P; ++c) {
          carry_hi[c] += carry_lo[c];
          carry_lo[c] = 0.f;
        }
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
// Tiles of a row are numbered k = 0, 1, ... from the right end (scan order),
// A(k) is tile k's sum, and tiles are grouped 32-ary: node(0, m) = A(m) and
// node(L+1, m) is the sum of node(L, 32m .. 32m+31), added with a fixed
// pairwise tree (adjacent pairs first).  Writing k in base 32, the tiles to
// the right of tile k are exactly, for every level L, the siblings that
// precede k's level-L ancestor under the same parent, so
//     E(k) = sum over L (from 0 up) of tree(node(L, first_L .. first_L + d_L - 1)),
// d_L being k's base-32 digit L.  Warp L reads the d_L siblings of level L in
// one round trip (all levels at once) and adds them with the same fixed tree,
// so E(k) never depends on timing and reruns are bit-identical.
//
// Publication needs no atomics: every tile publishes A(k); a tile whose level-L
// ancestor is the last child of its parent (digits 0..L all 31) has read the
// other 31 children, so it publishes the parent.  Values are 64-bit words
// {epoch, fp32 bits} written and read with relaxed single-copy-atomic
// accesses; a word counts only if its epoch is this launch's.
//
// Forward progress: tickets are taken in scan order and every node a tile
// waits for is published by a tile with a smaller ticket, whose block is
// already running and itself waits only on smaller tickets.  Every wait is
// bounded; when one runs out the block records the failure (error word, plus
// this launch's epoch in the abort word so the other waiters stop early) and
// finishes.
// ---------------------------------------------------------------------------
constexpr int kMaxLevels = kNW;  // one warp per level: 32^8 tiles per row at most



template <int VEC, int SUB>
__global__ void __launch_bounds__(kThreads, 3) k_rscan_lookback(RScanLookbackParams p) {
  pdl_begin();
  constexpr int64_t TILE = (int64_t)SUB * kThreads * VEC;
  __shared__ float sh_w[SUB][kNW][1];
  __shared__ float s_part[kMaxLevels];
  __shared__ unsigned s_ticket, s_epoch;
  __shared__ int s_fail;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int w = t >> 5;
  const unsigned* abort_word = p.err_word + 1;

  if (t == 0) {
    const Ticket tk = take_ticket(p.ticket_word);
    s_ticket = tk.ticket;
    s_epoch = tk.epoch;
    s_fail = 0;
    // Every other ticket is taken before the last one: reset for the next launch.
    if ((int64_t)tk.ticket == p.rows * p.tiles_per_row - 1) next_launch(p.ticket_word, tk.epoch);
  }
  __syncthreads();
  const int64_t ticket = s_ticket;
  const unsigned epoch = s_epoch;
  const int64_t tiles = p.tiles_per_row;
  if (ticket >= p.rows * tiles) {  // a stale counter: touch nothing
    if (t == 0) atomicOr(p.err_word, 2u);
    return;
  }
  const int64_t row = ticket / tiles;
  const int64_t k = ticket - row * tiles;       // from the right
  const int64_t base = (tiles - 1 - k) * TILE;  // tiles are aligned at the row's left end
  unsigned long long* vals = p.node_val + row * 2 * tiles;
  const bool stalled = ticket == p.stall_tile;

  const bool mirror = (p.flags & kScanMirror) != 0;
  const TileView tv = tile_view(row_view<VEC>(p.x, p.y, row, p.N), base, TILE, mirror);
  float v[SUB][VEC];
  load_tile<VEC, SUB>(v, tv, t, mirror);
  mask_tile<VEC, SUB>(v, tv, t, mirror);
  const TileScan<SUB> ts = tile_suffix<VEC, SUB>(v, sh_w, lane, w);
  if (t == 0 && !stalled) st_relaxed_u64(vals + k, pack_node(epoch, ts.total[0]));

  // Levels of this row: base-32 digits of the largest tile index.
  int levels = 1;
  while (levels < kMaxLevels && ((tiles - 1) >> (5 * levels)) != 0) ++levels;

  // Warp L reads the level-L siblings that precede k's ancestor (all levels
  // at once).  Warp 0 also publishes every parent this tile completes, right
  // after the read of the level below it, so no publication waits on a level
  // it does not need.
  if (w < levels) {
    int64_t off = 0, count = tiles;
    for (int q = 0; q < w; ++q) {
      off += count;
      count >>= 5;
    }
    int64_t m = k >> (5 * w);
    int d = (int)(m & 31);
    bool fail = false;
    float sib = 0.f;
    if (lane < d) sib = wait_node(vals + off + (m - d) + lane, epoch, p.spin_limit, abort_word, &fail);
    const float part = warp_tree_adjacent(sib);
    if (lane == 0) s_part[w] = part;
    if (w == 0) {
      float own = ts.total[0];
      int L = 0;
      while (d == 31 && !stalled && !__any_sync(kFullMask, fail)) {
        const float parent = warp_tree_adjacent(lane < 31 ? sib : own);
        own = __shfl_sync(kFullMask, parent, 0);
        const int64_t next_off = off + count;
        if (lane == 0) st_relaxed_u64(vals + next_off + (m >> 5), pack_node(epoch, own));
        if (++L >= levels) break;
        off = next_off;
        count >>= 5;
        m >>= 5;
        d = (int)(m & 31);
        if (d != 31) break;  // the next parent is not complete yet: someone else's job
        sib = 0.f;
        if (lane < 31) sib = wait_node(vals + off + (m - 31) + lane, epoch, p.spin_limit, abort_word, &fail);
      }
    }
    if (__any_sync(kFullMask, fail) && lane == 0) s_fail = 1;
  }
  __syncthreads();

  if (t == 0) {
    float excl = 0.f;
    for (int L = 0; L < levels; ++L) excl += s_part[L];  // from the lowest level up
    s_part[0] = excl;
    if (s_fail) {
      atomicOr(p.err_word, 1u);
      atomicExch(p.err_word + 1, epoch);
    }
  }
  __syncthreads();
  finalize<VEC, SUB>(v, ts, s_part[0], (p.flags & kScanExclusive) != 0);
  store_tile<VEC, SUB>(v, tv, t, mirror);
}

// ---------------------------------------------------------------------------
// Look-back with the two touches of each tile a fixed number of tickets apart.
//
// A block with ticket t (one block per ticket, tickets 0 .. tiles + lag - 1)
//   1. starts a bulk copy (TMA engine) of tile t from HBM into shared memory;
//   2. meanwhile writes out tile u = t - lag: looks back for u's exclusive
//      suffix, which every tile to its right published about `lag` tickets
//      ago, rereads u (read from HBM only about lag * 32 KiB ago, so normally
//      served from L2), scans it and stores it;
//   3. sums tile t from shared memory and publishes the sum, completing
//      parents as the one-tile-per-block form does.
// The look-back rarely waits, the HBM read of tile t overlaps step 2, and HBM
// still sees each element read once and written once while the lag's tiles
// stay in L2.  Every wait is on a smaller ticket, so forward progress holds as
// in the other forms.  EARLY takes the steps as 1, reread of u, 3, then the
// rest of 2: the sum of tile t is out as soon as its copy lands, so a shorter
// lag suffices.  Measured on one row of 1e9: the reverse scan is faster in
// the plain order (96% of copy bandwidth against 94%), the forward (mirrored)
// scan with EARLY (92% against 85%).
// ---------------------------------------------------------------------------
//
// With P > 1 the row is a narrow plane of P columns read flat (see
// tile_suffix): every tile publishes P node words, one per class (node (L, m)
// of class c at word (off_L + m)*P + c), and every sum above is taken per
// class.
template <int SUB, bool EARLY, bool EDGES, int P = 1>
__global__ void __launch_bounds__(kThreads, P == 1 ? 4 : 3) k_rscan_lookback_l2(RScanLookbackParams p) {
  pdl_begin();
  constexpr int64_t TILE = (int64_t)SUB * kThreads * 4;
  __shared__ __align__(128) float s_tile[TILE];
  __shared__ unsigned long long s_bar;
  __shared__ float sh_w[SUB][kNW][P];
  __shared__ float s_red[kNW][P];
  __shared__ float s_part[kMaxLevels][P];
  __shared__ unsigned s_ticket, s_epoch;
  __shared__ int s_fail;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int w = t >> 5;
  const unsigned* abort_word = p.err_word + 1;
  const int64_t tiles = p.tiles_per_row;
  const int64_t total = p.rows * tiles;

  if (t == 0) {
    const Ticket tkt = take_ticket(p.ticket_word);
    const unsigned tk = tkt.ticket;
    s_ticket = tk;
    s_epoch = tkt.epoch;
    s_fail = 0;
    // Every other ticket is taken before the last one: reset for the next launch.
    if ((int64_t)tk == total + p.lag - 1) next_launch(p.ticket_word, tkt.epoch);
    if (tk < total) {
      const int64_t row = tk / tiles;
      const int64_t k = tk - row * tiles;
      const TileView tv = tile_view(row_view<4, EDGES>(p.x, nullptr, row, p.N), (tiles - 1 - k) * TILE, TILE,
                                    (p.flags & kScanMirror) != 0);
      if (!EDGES || tv.len > 0) {  // 0: a tile past this row's end
        mbar_init(&s_bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&s_bar, (unsigned)tv.len * 4u);
        bulk_load(s_tile, tv.x, (unsigned)tv.len * 4u, &s_bar);
      }
    }
  }
  __syncthreads();
  const int64_t ticket = s_ticket;
  const unsigned epoch = s_epoch;
  if (ticket >= total + p.lag) {  // a stale counter: touch nothing
    if (t == 0) atomicOr(p.err_word, 2u);
    return;
  }
  int levels = 1;
  while (levels < kMaxLevels && ((tiles - 1) >> (5 * levels)) != 0) ++levels;

  // ---- reread tile `ticket - lag` (from L2), in flight while tile `ticket` lands ----
  const int64_t u = ticket - p.lag;
  const bool mirror = (p.flags & kScanMirror) != 0;
  float v[SUB][4];
  TileView tv_u{};
  if (u >= 0) {
    const int64_t row = u / tiles;
    const int64_t k = u - row * tiles;
    tv_u = tile_view(row_view<4, EDGES>(p.x, p.y, row, p.N), (tiles - 1 - k) * TILE, TILE, mirror);
    load_tile<4, SUB>(v, tv_u, t, mirror);
  }

  // ---- write out tile `ticket - lag` ----
  const auto write_out = [&]() {
    if (u < 0) return;
    const int64_t row = u / tiles;
    const int64_t k = u - row * tiles;
    unsigned long long* vals = p.node_val + row * 2 * tiles * P;
    if (w < levels) {
      int64_t off = 0, count = tiles;
      for (int q = 0; q < w; ++q) {
        off += count;
        count >>= 5;
      }
      const int64_t m = k >> (5 * w);
      const int d = (int)(m & 31);
      bool fail = false;
      float sib[P];
#pragma unroll
      for (int c = 0; c < P; ++c) sib[c] = 0.f;
      if (lane < d) {
        if constexpr (P == 1)
          sib[0] = wait_node(vals + off + (m - d) + lane, epoch, p.spin_limit, abort_word, &fail);
        else
          wait_node_classes<P>(vals + (off + (m - d) + lane) * P, epoch, p.spin_limit, abort_word, &fail, sib);
      }
#pragma unroll
      for (int c = 0; c < P; ++c) {
        const float part = warp_tree_adjacent(sib[c]);
        if (lane == 0) s_part[w][c] = part;
      }
      if (__any_sync(kFullMask, fail) && lane == 0) s_fail = 1;
    }
    if constexpr (EDGES) mask_tile<4, SUB>(v, tv_u, t, mirror);
    // The tile scan's barrier publishes s_part; each class's carry is its
    // look-back partials from the lowest level up.
    const auto excl_of = [&](int c) {
      float excl = 0.f;
      for (int L = 0; L < levels; ++L) excl += s_part[L][c];
      return excl;
    };
    if constexpr (P == 1) {
      const TileScan<SUB, P> ts = tile_suffix<4, SUB, P>(v, sh_w, lane, w);
      finalize<4, SUB>(v, ts, excl_of(0), (p.flags & kScanExclusive) != 0);
    } else {
      float unused[P];
      tile_scan_apply<4, SUB, P>(v, sh_w, lane, w, excl_of, (p.flags & kScanExclusive) != 0, unused);
    }
    store_tile<4, SUB, EDGES>(v, tv_u, t, mirror);
  };

  // The reverse scan writes first (its reread overlaps tile `ticket`'s copy),
  // then publishes; the forward (mirrored) scan publishes as soon as its copy
  // lands and writes last (measured faster in each direction).
  if constexpr (!EARLY) write_out();
  // ---- sum tile `ticket` (in shared memory) and publish it ----
  if (ticket < total) {
    const int64_t row = ticket / tiles;
    const int64_t k = ticket - row * tiles;
    // The copy's layout: shared element jj is tv.x[jj], whatever the direction.
    const TileView tv = tile_view(row_view<4, EDGES>(p.x, nullptr, row, p.N), (tiles - 1 - k) * TILE, TILE,
                                  (p.flags & kScanMirror) != 0);
    // The copy of this tile (time-bounded wait, independent of the poll limit).
    if ((!EDGES || tv.len > 0) && !mbar_wait_copy(&s_bar, 0u)) s_fail = 1;
    // Class sums of the copied tile.  Shared element jj is memory element
    // jj of the tile; in scan order it is jj (reverse scan) or len-1-jj
    // (mirrored), so with P > 1 component c of a float4 is in class c % P,
    // or (3 - c) % P mirrored (len and jj are multiples of 4).  P == 1 sums
    // the sub-tiles by a tree; P > 1 adds them in order as they are read (a
    // fixed order too, and no SUB x P values held).
    float e[P == 1 ? SUB : 1][P];
    float a[P];
#pragma unroll
    for (int c = 0; c < P; ++c) a[c] = 0.f;
#pragma unroll
    for (int s = 0; s < SUB; ++s) {
      const int jj = s * kThreads * 4 + t * 4;
      float q[4] = {0.f, 0.f, 0.f, 0.f};
      if (jj < tv.len) {
        const float4 f = *reinterpret_cast<const float4*>(s_tile + jj);
        q[0] = f.x;
        q[1] = f.y;
        q[2] = f.z;
        q[3] = f.w;
        if (EDGES && tile_has_edge(tv) && (jj < tv.lo || jj + 4 > tv.hi)) {  // an edge of the row
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (jj + c < tv.lo || jj + c >= tv.hi) q[c] = 0.f;
        }
      }
      if constexpr (P == 1) {
        e[s][0] = (q[0] + q[1]) + (q[2] + q[3]);
      } else if constexpr (P == 2) {
        const float even = q[0] + q[2], odd = q[1] + q[3];
        a[0] += mirror ? odd : even;
        a[1] += mirror ? even : odd;
      } else {
        static_assert(P == 4, "P is 1, 2 or 4");
#pragma unroll
        for (int c = 0; c < 4; ++c) a[c] += mirror ? q[3 - c] : q[c];
      }
    }
    if constexpr (P == 1) {
      float ec[SUB];
#pragma unroll
      for (int s = 0; s < SUB; ++s) ec[s] = e[s][0];
      a[0] = tree_sum<SUB>(ec);
    }
    block_sum_p<P>(a, s_red);  // warp 0, lane 0
    unsigned long long* vals = p.node_val + row * 2 * tiles * P;
    const bool stalled = ticket == p.stall_tile;
    if (w == 0 && !stalled) {
      float own[P];
#pragma unroll
      for (int c = 0; c < P; ++c) own[c] = __shfl_sync(kFullMask, a[c], 0);
      if (lane < P) st_relaxed_u64(vals + k * P + lane, pack_node(epoch, pick_class<P>(own, lane)));
      if ((k & 31) == 31) {  // publish every parent this tile completes
        bool fail = false;
        int64_t off = 0, count = tiles, m = k;
        for (int L = 0; L < levels && (m & 31) == 31; ++L) {
          float sib[P];
#pragma unroll
          for (int c = 0; c < P; ++c) sib[c] = 0.f;
          if (lane < 31) {
            if constexpr (P == 1)
              sib[0] = wait_node(vals + off + (m - 31) + lane, epoch, p.spin_limit, abort_word, &fail);
            else
              wait_node_classes<P>(vals + (off + (m - 31) + lane) * P, epoch, p.spin_limit, abort_word, &fail, sib);
          }
          if (__any_sync(kFullMask, fail)) break;
#pragma unroll
          for (int c = 0; c < P; ++c) {
            const float parent = warp_tree_adjacent(lane < 31 ? sib[c] : own[c]);
            own[c] = __shfl_sync(kFullMask, parent, 0);
          }
          const int64_t next_off = off + count;
          if (lane < P)
            st_relaxed_u64(vals + (next_off + (m >> 5)) * P + lane, pack_node(epoch, pick_class<P>(own, lane)));
          off = next_off;
          count >>= 5;
          m >>= 5;
        }
        if (fail && lane == 0) s_fail = 1;
      }
    }
  }
  if constexpr (EARLY) write_out();
  __syncthreads();
  if (t == 0 && s_fail) {
    atomicOr(p.err_word, 1u);
    atomicExch(p.err_word + 1, epoch);
  }
}

// ---------------------------------------------------------------------------
// Reduce-then-scan along rows: the deterministic multi-pass alternative to the
// look-back (each element travels three times between HBM and the SMs instead
// of two).  Both tile passes address logical tile k of the (possibly
// mirrored) row, and the middle pass -- a reverse exclusive row scan of the
// tile sums -- turns the sums into each tile's carry.
// ---------------------------------------------------------------------------
template <int VEC, int SUB, bool EDGES>
__global__ void __launch_bounds__(kThreads) k_tile_sums(TileSumsParams p) {
  pdl_begin();
  constexpr int64_t TILE = (int64_t)SUB * kThreads * VEC;
  __shared__ float sh[kNW];
  const int64_t b = blockIdx.x;
  const int64_t row = b / p.tiles;
  const int64_t k = b - row * p.tiles;
  float v[SUB][VEC];
  const bool mirror = (p.flags & kScanMirror) != 0;
  const TileView tv = tile_view(row_view<VEC, EDGES>(p.x, nullptr, row, p.N), k * TILE, TILE, mirror);
  load_tile<VEC, SUB>(v, tv, threadIdx.x, mirror);
  if constexpr (EDGES) mask_tile<VEC, SUB>(v, tv, threadIdx.x, mirror);
  float e[SUB];
#pragma unroll
  for (int s = 0; s < SUB; ++s) e[s] = tree_sum<VEC>(v[s]);
  const float a = block_sum<kThreads>(tree_sum<SUB>(e), sh);
  if (threadIdx.x == 0) st_plain(p.sums + b, a);
}

template <int VEC, int SUB, bool EDGES>
__global__ void __launch_bounds__(kThreads, 3) k_tile_carry_scan(TileCarryParams p) {
  pdl_begin();
  constexpr int64_t TILE = (int64_t)SUB * kThreads * VEC;
  __shared__ float sh_w[SUB][kNW][1];
  const int t = threadIdx.x;
  const int64_t b = blockIdx.x;
  const int64_t row = b / p.tiles;
  const int64_t k = b - row * p.tiles;
  const bool mirror = (p.flags & kScanMirror) != 0;
  float v[SUB][VEC];
  const TileView tv = tile_view(row_view<VEC, EDGES>(p.x, p.y, row, p.N), k * TILE, TILE, mirror);
  load_tile<VEC, SUB>(v, tv, t, mirror);
  if constexpr (EDGES) mask_tile<VEC, SUB>(v, tv, t, mirror);
  const TileScan<SUB> ts = tile_suffix<VEC, SUB>(v, sh_w, t & 31, t >> 5);
  finalize<VEC, SUB>(v, ts, ld_plain(p.carries + b), (p.flags & kScanExclusive) != 0);
  store_tile<VEC, SUB, EDGES>(v, tv, t, mirror);
}

// ---------------------------------------------------------------------------
// Cumulative sum along a strided axis: x, y are [outer, N, inner] with
// inner > 1 (the POPCORNBENCH trace l1_p91 discusses scanning dims other than
// the last).  A block owns CW = WX*32*VEC adjacent columns of one (o, segment)
// and walks the segment in the scan direction in tiles of T = WY*U rows: warp
// row wy loads rows [wy*U, wy*U + U) of the tile (every warp load is 32*VEC
// consecutive floats of one row), scans them in registers, and publishes its
// U-row total in shared memory; each thread then adds the totals of the warp
// rows before its own (pre) and of all WY (the tile total) in a fixed order.
// Output = base + (pre + own prefix), with base the blocked running sum of
// the earlier tiles' totals (starting from the segment's carry), so no
// addition chain grows with N and no output subtracts anything.  Splitting
// the rows of a tile over WY warps gives every column WY threads and keeps
// U*VEC loads in flight per thread, with one barrier per tile.
// ---------------------------------------------------------------------------

template <int VEC, int WX, int WY, int U>
__global__ void __launch_bounds__(kThreads, VEC == 4 ? 3 : 4) k_scan_cols(ScanColsParams p) {
  pdl_begin();
  static_assert(WX * WY * 32 == kThreads, "WX warps across columns, WY down the axis");
  constexpr int CW = WX * 32 * VEC;
  constexpr int T = WY * U;
  __shared__ __align__(16) float sh[2][WY][CW];
  const int warp = threadIdx.x >> 5;
  const int wx = warp % WX;
  const int wy = warp / WX;
  const int jloc = (wx * 32 + (threadIdx.x & 31)) * VEC;
  const int64_t col_tiles = (p.inner + CW - 1) / CW;
  const int64_t units = p.outer * p.segs * col_tiles;
  const int64_t step_j = p.reverse ? -p.inner : p.inner;
  int buf = 0;
  for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int64_t og = unit / col_tiles;  // (o, segment)
    const int64_t col = (unit - og * col_tiles) * CW + jloc;
    const int64_t o = og / p.segs;
    const int64_t lo = (og - o * p.segs) * p.seg_len;
    const int64_t len = min(p.seg_len, p.N - lo);
    // With VEC == 4 the caller guarantees inner % 4 == 0: all four columns.
    const bool active = col < p.inner;
    const int64_t j0 = p.reverse ? lo + len - 1 : lo;
    const int64_t off = (o * p.N + j0) * p.inner + (active ? col : 0);
    const float* xp = p.x + off;
    float* yp = p.y + off;
    float init[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c)
      init[c] = (p.carry != nullptr && active) ? ld_plain(p.carry + og * p.carry_stride + col + c) : 0.f;
    TileCarry<VEC> tc(init);
    for (int64_t t0 = 0; t0 < len; t0 += T) {
      // The stride is hidden from the optimiser each tile: otherwise it hoists
      // all U row offsets out of the loop and holds them in registers.
      int64_t sj = step_j;
      asm volatile("" : "+l"(sj));
      const int64_t k0 = t0 + wy * U;  // this warp row's first row, in scan order
      const int cnt = active ? (int)max((int64_t)0, min((int64_t)U, len - k0)) : 0;
      float q[U][VEC];
      const float* xr = xp + k0 * sj;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (u < cnt) {
          if constexpr (VEC == 4) {
            const float4 f = ld_stream4(xr);
            q[u][0] = f.x;
            q[u][1] = f.y;
            q[u][2] = f.z;
            q[u][3] = f.w;
          } else {
            q[u][0] = ld_stream1(xr);
          }
        } else {
#pragma unroll
          for (int c = 0; c < VEC; ++c) q[u][c] = 0.f;
        }
        xr += sj;
      }
#pragma unroll
      for (int u = 1; u < U; ++u)
#pragma unroll
        for (int c = 0; c < VEC; ++c) q[u][c] += q[u - 1][c];
      if constexpr (VEC == 4)
        *reinterpret_cast<float4*>(&sh[buf][wy][jloc]) =
            make_float4(q[U - 1][0], q[U - 1][1], q[U - 1][2], q[U - 1][3]);
      else
        sh[buf][wy][jloc] = q[U - 1][0];
      __syncthreads();
      float pre[VEC], tot[VEC], b[VEC];
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        float r = 0.f;
        pre[c] = 0.f;
#pragma unroll
        for (int y = 0; y < WY; ++y) {
          if (y == wy) pre[c] = r;
          r += sh[buf][y][jloc + c];
        }
        tot[c] = r;
        b[c] = tc.base(c);
      }
      float* yr = yp + k0 * sj;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (u < cnt) {
          float out[VEC];
#pragma unroll
          for (int c = 0; c < VEC; ++c) {
            const float own = p.exclusive ? (u > 0 ? q[u - 1][c] : 0.f) : q[u][c];
            out[c] = b[c] + (pre[c] + own);
          }
          if constexpr (VEC == 4) {
            st_stream4(yr, make_float4(out[0], out[1], out[2], out[3]));
          } else {
            st_stream1(yr, out[0]);
          }
        }
        yr += sj;
      }
      tc.add(tot);
      buf ^= 1;
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

int64_t lookback_tile(int variant) {
  switch (variant) {
    case kLookbackV1: return 8 * kThreads * 1;
    case kLookbackV4:
    case kLookbackL2: return 8 * kThreads * 4;
    default: return 0;
  }
}

cudaError_t launch_rscan_rows(int variant, const RScanRowsParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  if (p.period != 1) {  // narrow planes read flat: float4 tiles of 4 sub-tiles
    if (variant != kRScanV4S4) return cudaErrorInvalidValue;
    const bool edges = (p.flags & kScanRowEdges) != 0;
    if (p.period == 2) {
      if (edges) launch_pdl(k_rscan_rows<4, 4, true, 2>, g, kThreads, 0, s, p);
      else launch_pdl(k_rscan_rows<4, 4, false, 2>, g, kThreads, 0, s, p);
    } else if (p.period == 4) {
      if (edges) launch_pdl(k_rscan_rows<4, 4, true, 4>, g, kThreads, 0, s, p);
      else launch_pdl(k_rscan_rows<4, 4, false, 4>, g, kThreads, 0, s, p);
    } else {
      return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
  }
  switch (variant) {
    case kRScanV1S4: launch_pdl(k_rscan_rows<1, 4, false>, g, kThreads, 0, s, p); break;
    case kRScanV4S2:
      if (p.flags & kScanRowEdges) launch_pdl(k_rscan_rows<4, 2, true>, g, kThreads, 0, s, p);
      else launch_pdl(k_rscan_rows<4, 2, false>, g, kThreads, 0, s, p);
      break;
    case kRScanV4S4:
      if (p.flags & kScanRowEdges) launch_pdl(k_rscan_rows<4, 4, true>, g, kThreads, 0, s, p);
      else launch_pdl(k_rscan_rows<4, 4, false>, g, kThreads, 0, s, p);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// Sub-tiles of the L2 look-back: 8 (8192-float tiles) for plain rows; 4 for
// planes read flat, whose per-class arrays would not fit the registers of 3
// blocks per SM at 8.
template <int P>
constexpr int kL2Sub = P == 1 ? 8 : 4;

template <int P>
cudaError_t launch_l2_p(const RScanLookbackParams& p, dim3 g, cudaStream_t s) {
  constexpr int SUB = kL2Sub<P>;
  if (p.flags & kScanRowEdges) {
    if (p.flags & kScanMirror) launch_pdl(k_rscan_lookback_l2<SUB, true, true, P>, g, kThreads, 0, s, p);
    else launch_pdl(k_rscan_lookback_l2<SUB, false, true, P>, g, kThreads, 0, s, p);
  } else {
    if (p.flags & kScanMirror) launch_pdl(k_rscan_lookback_l2<SUB, true, false, P>, g, kThreads, 0, s, p);
    else launch_pdl(k_rscan_lookback_l2<SUB, false, false, P>, g, kThreads, 0, s, p);
  }
  return cudaGetLastError();
}

cudaError_t launch_rscan_lookback(int variant, const RScanLookbackParams& p, int64_t grid,
                                  cudaStream_t s) {
  if (variant != kLookbackL2 && p.period != 1) return cudaErrorInvalidValue;
  const dim3 g((unsigned)grid);
  switch (variant) {
    case kLookbackV1: launch_pdl(k_rscan_lookback<1, 8>, g, kThreads, 0, s, p); break;
    case kLookbackV4: launch_pdl(k_rscan_lookback<4, 8>, g, kThreads, 0, s, p); break;
    case kLookbackL2:
      if (p.period == 2) return launch_l2_p<2>(p, g, s);
      if (p.period == 4) return launch_l2_p<4>(p, g, s);
      if (p.period != 1) return cudaErrorInvalidValue;
      return launch_l2_p<1>(p, g, s);
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

int occupancy_rscan_lookback(int variant) {
  switch (variant) {
    case kLookbackV1: return occupancy_of(k_rscan_lookback<1, 8>);
    case kLookbackV4: return occupancy_of(k_rscan_lookback<4, 8>);
    case kLookbackL2:
      return std::min({occupancy_of(k_rscan_lookback_l2<8, false, false>),
                       occupancy_of(k_rscan_lookback_l2<8, true, false>),
                       occupancy_of(k_rscan_lookback_l2<8, false, true>),
                       occupancy_of(k_rscan_lookback_l2<8, true, true>)});
    default: return 0;
  }
}

cudaError_t launch_scan_cols(int variant, const ScanColsParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  switch (variant) {
    case kScanColsV1: launch_pdl(k_scan_cols<1, 2, 4, 16>, g, kThreads, 0, s, p); break;
    case kScanColsV4: launch_pdl(k_scan_cols<4, 2, 4, 8>, g, kThreads, 0, s, p); break;
    case kScanColsV4Y8: launch_pdl(k_scan_cols<4, 1, 8, 8>, g, kThreads, 0, s, p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

int scan_cols_block_width(int variant) {
  switch (variant) {
    case kScanColsV1: return 2 * 32;
    case kScanColsV4: return 2 * 32 * 4;
    case kScanColsV4Y8: return 32 * 4;
    default: return 0;
  }
}

int scan_cols_tile_rows(int variant) {
  switch (variant) {
    case kScanColsV1: return 4 * 16;
    case kScanColsV4: return 4 * 8;
    case kScanColsV4Y8: return 8 * 8;
    default: return 0;
  }
}

int64_t tile_scan_len(int variant) { return variant == kTileV4 ? 8 * kThreads * 4 : 8 * kThreads; }

cudaError_t launch_tile_sums(int variant, const TileSumsParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  if (variant == kTileV4) {
    if (p.flags & kScanRowEdges) launch_pdl(k_tile_sums<4, 8, true>, g, kThreads, 0, s, p);
    else launch_pdl(k_tile_sums<4, 8, false>, g, kThreads, 0, s, p);
  } else {
    launch_pdl(k_tile_sums<1, 8, false>, g, kThreads, 0, s, p);
  }
  return cudaGetLastError();
}

cudaError_t launch_tile_carry_scan(int variant, const TileCarryParams& p, int64_t grid, cudaStream_t s) {
  const dim3 g((unsigned)grid);
  if (variant == kTileV4) {
    if (p.flags & kScanRowEdges) launch_pdl(k_tile_carry_scan<4, 8, true>, g, kThreads, 0, s, p);
    else launch_pdl(k_tile_carry_scan<4, 8, false>, g, kThreads, 0, s, p);
  } else {
    launch_pdl(k_tile_carry_scan<1, 8, false>, g, kThreads, 0, s, p);
  }
  return cudaGetLastError();
}

int occupancy_scan_cols(int variant) {
  switch (variant) {
    case kScanColsV1: return occupancy_of(k_scan_cols<1, 2, 4, 16>);
    case kScanColsV4: return occupancy_of(k_scan_cols<4, 2, 4, 8>);
    case kScanColsV4Y8: return occupancy_of(k_scan_cols<4, 1, 8, 8>);
    default: return 0;
  }
}

// Narrow planes read flat (period 2 or 4): the L2 look-back and the float4
// block-per-row kernel.
template <int P>
int occupancy_l2_p() {
  constexpr int SUB = kL2Sub<P>;
  return std::min({occupancy_of(k_rscan_lookback_l2<SUB, false, false, P>),
                   occupancy_of(k_rscan_lookback_l2<SUB, true, false, P>),
                   occupancy_of(k_rscan_lookback_l2<SUB, false, true, P>),
                   occupancy_of(k_rscan_lookback_l2<SUB, true, true, P>)});
}
int occupancy_rscan_lookback_period(int period) {
  if (period == 2) return occupancy_l2_p<2>();
  if (period == 4) return occupancy_l2_p<4>();
  return occupancy_rscan_lookback(kLookbackL2);
}
int64_t lookback_tile_period(int period) { return (int64_t)(period == 1 ? kL2Sub<1> : kL2Sub<2>) * kThreads * 4; }
int occupancy_rscan_rows_period(int period) {
  if (period == 2) return std::min(occupancy_of(k_rscan_rows<4, 4, false, 2>), occupancy_of(k_rscan_rows<4, 4, true, 2>));
  if (period == 4) return std::min(occupancy_of(k_rscan_rows<4, 4, false, 4>), occupancy_of(k_rscan_rows<4, 4, true, 4>));
  return occupancy_rscan_rows(kRScanV4S4);
}

int occupancy_rscan_rows(int variant) {
  switch (variant) {
    case kRScanV1S4: return occupancy_of(k_rscan_rows<1, 4, false>);
    case kRScanV4S2: return std::min(occupancy_of(k_rscan_rows<4, 2, false>), occupancy_of(k_rscan_rows<4, 2, true>));
    case kRScanV4S4: return std::min(occupancy_of(k_rscan_rows<4, 4, false>), occupancy_of(k_rscan_rows<4, 4, true>));
    default: return 0;
  }
}

}  // namespace lr
