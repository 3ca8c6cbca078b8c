// lr_internal.h -- kernel parameter blocks and launchers shared between the
// C-ABI layer (lr_api.cu) and the kernel translation units.  Not installed.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace lr {

// Launch `kernel` with programmatic stream serialization (see pdl_begin in
// lr_device.cuh: the kernel waits for its predecessor before touching memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, unsigned block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}


// Output epilogue of the reduce kernels: the mean divides the sum by the
// element count, the norm takes the square root of the sum of squares.
enum Epilogue { kEpiNone = 0, kEpiMean = 1, kEpiSqrt = 2 };

constexpr int kThreads = 256;  // every libreduce kernel runs 256-thread blocks

// --- 1D sum and row sums over contiguous segments --------------------------
// Segment g is x[g*seg_len, (g+1)*seg_len).  Each segment is cut into
// `chunks` chunks of chunk_len elements (the last may be shorter); block b
// reduces chunk (b % chunks) of segment (b / chunks).  With chunks > 1 the
// block partials go to `partials` and the last block of a segment (picked by
// an integer ticket) sums them in chunk order.
struct ContigParams {
  const float* x;
  int64_t seg_len;
  int64_t chunk_len;  // multiple of 4
  int32_t chunks;
  float* out;          // one float per segment
  float* partials;     // segments * chunks floats (chunks > 1)
  unsigned* tickets;   // one per segment, zero on entry, left zero on exit
  int epi;             // output epilogue (kEpiNone, kEpiMean, kEpiSqrt)
};

// --- 1D reduction of a short array by one thread-block cluster ---------------
// CTA r of a cluster of `chunks` CTAs (kClusterThreads threads each) reduces
// x[r*chunk_len, min((r+1)*chunk_len, seg_len)) with all of its loads in
// flight at once; CTA 0 combines the CTAs' results in rank order through
// distributed shared memory and writes out[0].  No scratch, no ticket, one
// launch.  The host keeps chunk_len <= kClusterThreads * kClusterLoads * 4.
constexpr int kClusterThreads = 512;
constexpr int kClusterLoads = 16;   // float4 loads per thread
constexpr int kClusterMaxCtas = 8;  // the portable cluster size
constexpr int64_t kClusterMaxN = (int64_t)kClusterMaxCtas * kClusterThreads * kClusterLoads * 4;  // 2^18

// --- Row sums, one warp per row (short rows) -------------------------------
struct RowsWarpParams {
  const float* x;
  int64_t rows;
  int64_t len;
  float* out;
  int epi;
};

// --- Axis sum with inner > 1 ------------------------------------------------
// Block b covers column tile ct = b % col_tiles, reduce slice s = (b /
// col_tiles) % splits and outer index o = b / (col_tiles * splits).  With
// splits > 1 each block writes its column sums to partials[(o*splits + s) *
// col_tiles * CW + ct * CW + j] and the last block of (o, ct) sums the slices
// in slice order.
struct ColsParams {
  const float* x;
  int64_t outer, reduce, inner;
  int32_t col_tiles;
  int32_t splits;
  int64_t rows_per_split;
  float* out;
  float* partials;
  unsigned* tickets;  // outer * col_tiles, zero on entry, left zero on exit
  int epi;
  int keep_partials;  // split only: leave every slice's column sums in `partials`
};

// --- Scan flags (internal) ---------------------------------------------------
// The row kernels compute a reverse (suffix) scan; a forward scan is the
// reverse scan of the mirrored row (kScanMirror), and an exclusive scan leaves
// out each element's own term (kScanExclusive).
constexpr int kScanMirror = 1;
constexpr int kScanExclusive = 2;
// Set by the host for float4 row scans whose rows are not whole aligned
// float4s (N % 4 != 0 or x not 16-byte aligned): selects the kernel form that
// masks the row edges.
constexpr int kScanRowEdges = 4;

// --- Cumulative sum along rows, one block per row ----------------------------
// period P (1, 2 or 4): the row is a narrow plane of P columns read flat,
// element e in column class e % P, and each class is scanned on its own
// (float4 tiles only).
struct RScanRowsParams {
  const float* x;
  float* y;
  int64_t rows;
  int64_t N;
  int flags;
  int period = 1;
};

// --- Scans of many short rows (N <= kShortRowMax) -----------------------------
// A block stages a chunk of rows_per_chunk whole rows in shared memory (row r
// of the chunk at r*stride floats), scans each row with a group of `lanes`
// lanes (a power of two, 1..32; the kernel's template parameter), each lane
// taking a run of run_len consecutive elements, and stores the chunk back.
// magic = ceil(2^32 / N): the row of flat index e of a chunk is
// (e*magic) >> 32, exact for every e < kShortSmem and N <= 4096.
constexpr int kShortRowMax = 2048;    // longest row this form takes
constexpr int kShortChunk = 3072;     // data floats per chunk (about; at least 8 rows where they fit)
constexpr int kShortSmem = 6144;      // shared floats per block (24 KB)
constexpr int kShortThreads = 128;    // threads per block
// Load forms of the short-row kernels (the launchers' `vec`):
constexpr int kShortLd1 = 1;  // 4-byte loads (any 4-byte alignment)
constexpr int kShortLd4 = 4;  // 16-byte loads; every row is whole float4s (N % 4 == 0)
//
// Narrow planes (inner > 1): x is [rows, N, inner] -- `rows` planes of N rows
// of `inner` columns -- and every (plane, column) is scanned or reduced along
// N.  A chunk holds rows_per_chunk whole planes; it is staged transposed, so
// column c of the chunk's plane q is the shared-memory row q*inner + c (of N
// elements, at (q*inner + c)*stride), and the row code above runs unchanged.
// magic_inner = ceil(2^32 / inner) divides a flat plane index by inner
// (exact for every index below kShortSmem and inner <= 4096).
struct ShortRowsParams {
  const float* x;
  float* y;
  int64_t rows;
  int N;
  int rows_per_chunk;
  int stride;
  int run_len;
  unsigned long long magic;
  int flags;  // kScanMirror | kScanExclusive
  int inner;  // 1: plain rows; > 1: narrow planes
  unsigned long long magic_inner;
};

// --- Narrow planes of 2-8 columns, read flat (segmented class runs) -----------
// x is [outer, N, P] (P = 2 .. kPlanesMaxP columns), scanned or reduced along N.
// Plane o is the L = N*P floats from o*L; the float at flat index f is in
// column f % P.  Work is cut into items of k whole planes: k >= 2 planes fit
// one tile of planes_tile_len(P) floats (with the item's start rounded down
// to planes_align(P)); k = 1 covers a plane in one or more tiles.  x (and y
// for scans) must be 16-byte aligned and N >= 2 (with L <= planes_run_len(P)
// the kernels take the form for several plane boundaries in one thread's run).
constexpr int kPlanesThreads = 128;  // threads per block (these kernels only)
constexpr int kPlanesMaxP = 8;       // columns of every form: 2 .. kPlanesMaxP
constexpr int kPlanesMaxScanP = 14;  // the runs also scan 9, 10, 12 and 14 columns
__host__ __device__ constexpr bool planes_scan_columns(int P) {
  return (P >= 2 && P <= kPlanesMaxP) || P == 9 || P == 10 || P == 12 || P == 14;
}
// Scans as column groups (k_planes_cg), 3 .. kPlanesCgMaxP columns: thread t
// owns column group t % G of a run of planes_cg_run_rows rows, a group being
// V = planes_cg_vec(P) adjacent columns (a float4, float2 or float) and G =
// P / V <= 32; 128 / G row groups of a run make a tile of
// planes_cg_tile_rows(P) whole rows.  Runs of 9, 17 and 33 rows (1 modulo
// 32 / gcd(P, 32)) put the threads of a shared-memory phase on distinct
// banks.  Planes of more than one run (N > planes_cg_run_rows).
constexpr int kPlanesCgMaxP = 128;
__host__ __device__ constexpr int planes_cg_vec(int P) { return P % 4 == 0 ? 4 : P % 2 == 0 ? 2 : 1; }
__host__ __device__ constexpr int planes_cg_run_rows_v(int V) { return V == 4 ? 9 : V == 2 ? 17 : 33; }
__host__ __device__ constexpr int planes_cg_run_rows(int P) { return planes_cg_run_rows_v(planes_cg_vec(P)); }
__host__ __device__ constexpr int planes_cg_groups(int P) { return P / planes_cg_vec(P); }
__host__ __device__ constexpr bool planes_cg_fits(int P) {
  return P >= 3 && P <= kPlanesCgMaxP && planes_cg_groups(P) <= 32;
}
__host__ __device__ constexpr int planes_cg_tile_rows(int P) {
  return kPlanesThreads / planes_cg_groups(P) * planes_cg_run_rows(P);
}
// The automatic choice and the plane-run option take the column groups for
// scans of 6 columns and more and reductions of 3 and of 5 columns and more
// (ahead of the runs there: measured), the runs for the rest and for planes
// no longer than a column-group run.
__host__ __device__ constexpr bool planes_cg_scan(int P) { return planes_cg_fits(P) && P >= 6; }
__host__ __device__ constexpr bool planes_cg_reduce(int P) { return planes_cg_fits(P) && (P == 3 || P >= 5); }
// Consecutive floats per thread (whole rows of P columns, at most 36), the
// alignment of runs and tiles (lcm(4, P) floats: 16 bytes and P), and floats
// per tile.
__host__ __device__ constexpr int planes_run_len(int P) {
  return P == 5 || P == 10 ? 20 : P == 7 || P == 14 ? 28 : P == 8 ? 24 : 36;
}
__host__ __device__ constexpr int planes_align(int P) {
  return P == 3 || P == 6 || P == 12 ? 12 : P == 5 ? 20 : P == 7 ? 28 : P == 8 ? 8 : P == 9 ? 36 : P == 10 ? 20
       : P == 14 ? 28 : 4;
}
__host__ __device__ constexpr int planes_tile_len(int P) { return kPlanesThreads * planes_run_len(P); }
struct PlaneRunParams {
  const float* x;
  float* y;            // scans: [outer, N, P]; reductions: [outer, P]
  int64_t outer;
  int64_t N;
  int64_t k;           // planes per item
  int64_t items;       // ceil(outer / k)
  unsigned long long magic;  // ceil(2^32 / L) when k >= 2 (then L < planes_tile_len(P) / 2)
  int flags;           // scans: kScanMirror | kScanExclusive; reductions: the epilogue
  unsigned* err_word;  // bit 0 set if a tile's copy never lands
  int multi = 0;       // planes of 2P .. planes_run_len(P) floats: several boundaries in a run
  int P = 0;           // columns (the column-group kernels take them at run time)
};

// Scans of few long planes of 2-8 columns, a plane's tiles spread over
// blocks: scan-order tile j of plane o is ticket o * tiles + j, and each
// tile's P class sums go through the deterministic 32-ary look-back of the
// row scans (node words {epoch, fp32}, class c of node (L, m) of plane o at
// word (o * 2 * tiles + off_L + m) * P + c).  tiles is the most tiles any
// plane covers; a plane with one fewer publishes an empty last tile.
constexpr int kPlanesLbLevels = kPlanesThreads / 32;  // one warp per level: 32^4 tiles per plane at most
struct PlaneLbParams {
  const float* x;
  float* y;
  int64_t outer, N;
  int64_t tiles;                    // tiles per plane
  unsigned long long* node_val;     // outer * 2 * tiles * P words
  unsigned long long* ticket_word;  // as in RScanLookbackParams
  unsigned* err_word;               // as in RScanLookbackParams
  int64_t spin_limit;               // polls before a wait gives up
  int64_t stall_tile;               // test fault: this ticket never publishes (-1: none)
  int64_t lag;                      // tickets between a tile's two touches
  int flags;                        // kScanMirror | kScanExclusive
  int P = 0;                        // columns (the column-group form takes them at run time)
};

// --- Reduce-then-scan along rows (three passes) ------------------------------
// Rows are scanned as reverse scans of the (possibly mirrored) row, in logical
// tiles k = [k*TILE, (k+1)*TILE).  Pass 1 writes the sum of every logical tile
// (sums[r*tiles + k]); pass 2 is a reverse exclusive row scan of those sums,
// giving each tile's carry (the sum of the tiles after it); pass 3 scans each
// tile again and adds its carry.  `flags` as for the row scans.
struct TileSumsParams {
  const float* x;
  int64_t rows, N, tiles;
  float* sums;
  int flags;
};
struct TileCarryParams {
  const float* x;
  float* y;
  int64_t rows, N, tiles;
  const float* carries;  // [rows, tiles], logical tile order
  int flags;
};

// --- Axis reduction over narrow rows (inner <= 32 column groups of VEC) -----
// x: [outer, reduce, inner]; one block per (o, slice).  With splits > 1 each
// slice's column values go to partials[(o*splits + s)*part_stride + c] and the
// last block of o (ticket) combines them, unless keep_partials is set.
struct NarrowParams {
  const float* x;
  int64_t outer, reduce, inner;
  int64_t splits, rows_per_split;
  float* out;
  float* partials;
  int64_t part_stride;
  unsigned* tickets;  // outer, zero on entry, left zero on exit
  int epi;
  int keep_partials;
};

// --- Cumulative sum along a strided axis (inner > 1) -------------------------
// x, y: [outer, N, inner]; one block per (o, segment, column tile).
struct ScanColsParams {
  const float* x;
  float* y;
  int64_t outer, N, inner;
  int reverse;
  int exclusive;
  // Segmented form (the last pass of a column reduce-then-scan): the axis is
  // cut into `segs` segments of seg_len rows, each scanned from
  // carry[(o*segs + s)*carry_stride + col].
  const float* carry;  // null: one segment, starting from zero
  int64_t segs, seg_len, carry_stride;
};

// --- Reverse cumulative sum, single-pass decoupled look-back ----------------
// One block per tile.  Blocks take tickets in scan order (right to left within
// a row, row after row): ticket t is tile k = t % tiles_per_row counted from
// the right end of row t / tiles_per_row.  Tile sums and 32-ary group sums are
// published as 64-bit words {epoch, fp32 bits}; a word counts only if its
// epoch equals this launch's, so the flags never need clearing.
struct RScanLookbackParams {
  const float* x;
  float* y;
  int64_t rows;
  int64_t N;
  int64_t tiles_per_row;
  unsigned long long* node_val;  // rows * 2 * tiles_per_row words
  unsigned long long* ticket_word;  // {epoch:32, ticket counter:32}; counter zero on entry,
                                   // reset (epoch advanced) by the block with the last ticket
  unsigned* err_word;              // bit 0 set when a wait runs out
  int64_t spin_limit;            // polls before a wait gives up
  int64_t stall_tile;            // test fault: this ticket never publishes (-1: none)
  int64_t lag;                   // L2-lag form: tiles between a tile's two touches
  int flags;                     // kScanMirror | kScanExclusive
  int period = 1;                // as in RScanRowsParams (L2-lag form only); node words x period
};

// --- Scan along a strided axis, single-pass look-back over column tiles -----
// x, y are [outer, N, inner], scanned along N.  A unit is (o, column tile ct)
// of kColLbCols columns; its tile k holds scan positions [k*kColLbRows,
// (k+1)*kColLbRows) (position n is row N-1-n when reverse).  Tickets run over
// (o, k, ct) with ct fastest, so blocks in flight cover whole rows.  Node
// words {epoch, fp32} per column: unit u's level-L node m, column c, is
// node_val[((u*2*tiles) + off_L + m) * kColLbCols + c].
constexpr int kColLbWarps = 8;                // warps per block; a warp covers 32 rows of a tile
constexpr int kColLbRows = 32 * kColLbWarps;  // rows per tile
constexpr int kColLbCols = 32;
constexpr int kColLbMaxLevels = 3;  // 32^3 tiles per unit at most
struct ScanColsLookbackParams {
  const float* x;
  float* y;
  int64_t outer, N, inner;
  int64_t col_tiles;                // ceil(inner / kColLbCols)
  int64_t tiles;                    // per unit: ceil(N / kColLbRows)
  unsigned long long* node_val;     // outer * col_tiles * 2 * tiles * kColLbCols words
  unsigned long long* ticket_word;  // as in RScanLookbackParams
  unsigned* err_word;               // as in RScanLookbackParams
  int64_t spin_limit;
  int64_t stall_tile;               // test fault: this ticket never publishes (-1: none)
  int64_t lag;                      // tickets between a tile's two touches
  int reverse, exclusive;
};

// Reduction operators of the reduce kernels (the epilogue in the params turns
// a sum into a mean and a sum of squares into a norm).
enum ReduceOp { kOpSum = 0, kOpSumSq = 1, kOpMax = 2, kOpMin = 3, kNumReduceOps };

// Variants are small integers chosen by the dispatcher; each launcher
// returns cudaErrorInvalidValue for a variant it does not have.  Operators
// other than kOpSum exist for the default variants only (kContigU16,
// kColsV1W4, kColsV4W4).
enum ContigVariant { kContigU4 = 0, kContigU8 = 1, kContigU16 = 2, kNumContigVariants };
enum ColsVariant {
  kColsV1W1 = 0,   // scalar columns, 8 warps across columns
  kColsV1W4 = 1,   // scalar columns, 2 warps across x 4 along rows
  kColsV1W8 = 2,   // scalar columns, 8 warps along rows
  kColsV4W1 = 3,   // float4 columns, 8 warps across columns
  kColsV4W4 = 4,
  kColsV4W8 = 5,
  kNumColsVariants
};
// Option values (not kernel shapes of the enum above): the narrow-row kernel,
// block form (one block per (o, slice)) and warp form (one warp per o).
constexpr int kColsNarrow = kNumColsVariants;
constexpr int kColsNarrowWarp = kNumColsVariants + 1;
constexpr int kColsShortPlanes = kNumColsVariants + 2;  // chunks of whole narrow planes (short-row kernels)
constexpr int kColsPlaneRuns = kNumColsVariants + 3;    // narrow planes, segmented class runs (lr_planes.cuh)
enum RScanVariant { kRScanV1S4 = 0, kRScanV4S2 = 1, kRScanV4S4 = 2, kNumRScanVariants };
enum LookbackVariant {
  kLookbackV1 = 0,  // scalar items, one tile per block, tile kept in registers
  kLookbackV4 = 1,  // float4 items, one tile per block, tile kept in registers
  kLookbackL2 = 2,  // float4 items, ticket t sums tile t and writes tile t - lag (L2 reread)
  kNumLookbackVariants
};

// Column scan block shapes: VEC floats per thread, WX warps across columns,
// WY warps down the axis, U rows per warp per tile.
enum ScanColsVariant {
  kScanColsV1 = 0,    // VEC 1, WX 2, WY 4, U 16
  kScanColsV4 = 1,    // VEC 4, WX 2, WY 4, U 8 (needs inner % 4 == 0, aligned x, y)
  kScanColsV4Y8 = 2,  // VEC 4, WX 1, WY 8, U 8 (same)
  kNumScanColsVariants
};
inline bool scan_cols_vec4(int variant) { return variant == kScanColsV4 || variant == kScanColsV4Y8; }
// Option values: the narrow-row scan, block form (tiles in shared memory) and
// warp form (one warp per (o, segment)).
constexpr int kScanColsNarrow = kNumScanColsVariants;
constexpr int kScanColsNarrowWarp = kNumScanColsVariants + 1;
constexpr int kScanColsLookback = kNumScanColsVariants + 2;  // k_scan_cols_lookback
constexpr int kScanColsShortPlanes = kNumScanColsVariants + 3;  // chunks of whole narrow planes (short-row kernels)
constexpr int kScanColsPeriodRows = kNumScanColsVariants + 4;   // planes of 2 or 4 columns as flat rows
constexpr int kScanColsPlaneRuns = kNumScanColsVariants + 5;    // narrow planes, segmented class runs (lr_planes.cuh)
constexpr int kScanColsPlaneLookback = kNumScanColsVariants + 6;  // the same tiles, a plane over blocks (look-back)
enum TileScanVariant { kTileV1 = 0, kTileV4 = 1, kNumTileVariants };

// Elements per tile of the reduce-then-scan passes.
int64_t tile_scan_len(int variant);

// Elements per tile of each look-back variant.
int64_t lookback_tile(int variant);

// Columns covered by one block of a cols variant.
int cols_block_width(int variant);

// Columns and rows (in scan order) of one tile of a column scan variant.
int scan_cols_block_width(int variant);
int scan_cols_tile_rows(int variant);

cudaError_t launch_reduce_contig(int variant, int op, const ContigParams& p, int64_t grid,
                                 cudaStream_t s);
// One cluster of `ctas` CTAs (1..kClusterMaxCtas); p.chunks == ctas.
cudaError_t launch_reduce_cluster(int op, const ContigParams& p, int ctas, cudaStream_t s);
cudaError_t launch_reduce_rows_warp(int op, const RowsWarpParams& p, int64_t grid, cudaStream_t s);
cudaError_t launch_reduce_cols(int variant, int op, const ColsParams& p, int64_t grid, cudaStream_t s);
cudaError_t launch_fill(float* out, int64_t n, float value, cudaStream_t s);
cudaError_t launch_rscan_rows(int variant, const RScanRowsParams& p, int64_t grid, cudaStream_t s);
cudaError_t launch_rscan_lookback(int variant, const RScanLookbackParams& p, int64_t grid,
                                  cudaStream_t s);
cudaError_t launch_scan_cols(int variant, const ScanColsParams& p, int64_t grid, cudaStream_t s);
cudaError_t launch_tile_sums(int variant, const TileSumsParams& p, int64_t grid, cudaStream_t s);
// Narrow rows: vec is 1 or 4 (4 needs inner % 4 == 0 and 16-byte aligned x, y);
// inner <= 32 * vec.
cudaError_t launch_reduce_narrow(int vec, int op, const NarrowParams& p, int64_t grid, cudaStream_t s);
cudaError_t launch_scan_narrow(int vec, const ScanColsParams& p, int64_t grid, cudaStream_t s);
int occupancy_reduce_narrow(int vec, int op);
int occupancy_scan_narrow(int vec);
int64_t scan_narrow_tile_rows(int vec, int64_t inner);  // rows of one tile, in scan order
// Warp forms (one warp per (o, segment) / per o): eight units per block.
cudaError_t launch_scan_narrow_warp(int vec, const ScanColsParams& p, int64_t grid, cudaStream_t s);
int occupancy_scan_narrow_warp(int vec);
cudaError_t launch_reduce_narrow_warp(int vec, int op, const NarrowParams& p, int64_t grid, cudaStream_t s);
cudaError_t launch_tile_carry_scan(int variant, const TileCarryParams& p, int64_t grid, cudaStream_t s);
// lanes: 1, 2, 4, 8, 16 or 32; vec: 4 for float4 loads and stores (N % 4 == 0,
// x and y 16-byte aligned), else 1.
cudaError_t launch_rscan_short(int lanes, int vec, const ShortRowsParams& p, int64_t grid, cudaStream_t s);
// The same chunks for reductions of short rows: p.y receives one float per
// row and p.flags holds the epilogue (kEpiNone, kEpiMean, kEpiSqrt).  lanes:
// 1, 8, 16 or 32.
cudaError_t launch_reduce_short(int op, int lanes, int vec, const ShortRowsParams& p, int64_t grid, cudaStream_t s);
int occupancy_rscan_short();
cudaError_t launch_scan_cols_lookback(int vec, const ScanColsLookbackParams& p, int64_t grid, cudaStream_t s);
// Narrow planes read flat: P = 2 .. kPlanesMaxP; reductions take any ReduceOp.
cudaError_t launch_planes_scan(int P, const PlaneRunParams& p, int64_t grid, cudaStream_t s);
cudaError_t launch_planes_reduce(int P, int op, const PlaneRunParams& p, int64_t grid, cudaStream_t s);
int occupancy_planes(int P, bool scan);  // resident kPlanesThreads-thread blocks per SM
// Column groups (k_planes_cg): the instance a column count takes (0 .. 5, -1
// when none), its launch (p.P set) and its resident blocks per SM.
constexpr int kPlanesCgInstances = 6;
int cg_instance(int P);
cudaError_t launch_planes_cg(const PlaneRunParams& p, int64_t grid, cudaStream_t s);
int occupancy_planes_cg(int instance);
cudaError_t launch_planes_cg_reduce(int op, const PlaneRunParams& p, int64_t grid, cudaStream_t s);
int occupancy_planes_cg_reduce(int instance);
// Few long planes as column groups: tiles over blocks, carries by look-back.
cudaError_t launch_planes_cg_lookback(const PlaneLbParams& p, int64_t grid, cudaStream_t s);
int occupancy_planes_cg_lookback(int instance);
int occupancy_planes_reduce(int P);
cudaError_t launch_planes_lookback(int P, const PlaneLbParams& p, int64_t grid, cudaStream_t s);
int occupancy_planes_lookback(int P);

int occupancy_scan_cols_lookback();

// --- Debug builds (LR_DEBUG) -------------------------------------------------
// The address ranges a call's kernels may touch, registered by the host in
// g_lr_debug (defined in lr_api.cu) before the call's launches; the device
// helpers check every access against them and record what falls outside.
constexpr int kDbgRanges = 6;
constexpr unsigned kDbgGlobal = 1u;      // a global access outside every registered range
constexpr unsigned kDbgShared = 2u;      // a shared-memory index outside its buffer
constexpr unsigned kDbgMisaligned = 4u;  // a vector access not aligned to its width
struct LrDebug {
  unsigned long long lo[kDbgRanges], hi[kDbgRanges];
  unsigned flags;
  unsigned long long first_bad;
};
// Register up to kDbgRanges byte ranges [p[i], p[i] + bytes[i]) on stream s
// (debug builds; a no-op returning cudaSuccess otherwise).
cudaError_t dbg_register_ranges(cudaStream_t s, const void* const* p, const size_t* bytes, int n);

// Host helpers defined in lr_api.cu, for entry points in other files.
int check_device_buffer(const void* p, size_t bytes, int dev);  // a libreduce status
int record_cuda_error(cudaError_t e);                           // returns the CUDA status
void count_launch();

// Resident 256-thread blocks per SM for each kernel variant (0 on error).
int occupancy_reduce_contig(int variant, int op);
int occupancy_reduce_rows_warp(int op);
int occupancy_reduce_cols(int variant, int op);
int occupancy_rscan_rows(int variant);
int occupancy_rscan_lookback(int variant);
int occupancy_rscan_rows_period(int period);      // float4 block per row, period 1, 2 or 4
int occupancy_rscan_lookback_period(int period);  // L2-lag look-back, period 1, 2 or 4
int64_t lookback_tile_period(int period);         // its tile (floats) at that period
int occupancy_scan_cols(int variant);

}  // namespace lr
