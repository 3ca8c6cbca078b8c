// lr_internal.h -- kernel parameter blocks and launchers shared between the
// C-ABI layer (lr_api.cu) and the kernel translation units.  Not installed.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace lr {

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
};

// --- Row sums, one warp per row (short rows) -------------------------------
struct RowsWarpParams {
  const float* x;
  int64_t rows;
  int64_t len;
  float* out;
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
};

// --- Reverse cumulative sum, one block per row ------------------------------
struct RScanRowsParams {
  const float* x;
  float* y;
  int64_t rows;
  int64_t N;
};

// Variants are small integers chosen by the dispatcher; each launcher
// returns cudaErrorInvalidValue for a variant it does not have.
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
enum RScanVariant { kRScanV1S4 = 0, kRScanV4S2 = 1, kRScanV4S4 = 2, kNumRScanVariants };

// Columns covered by one block of a cols variant.
int cols_block_width(int variant);

cudaError_t launch_reduce_contig(int variant, const ContigParams& p, int64_t grid, cudaStream_t s);
cudaError_t launch_reduce_rows_warp(const RowsWarpParams& p, int64_t grid, cudaStream_t s);
cudaError_t launch_reduce_cols(int variant, const ColsParams& p, int64_t grid, cudaStream_t s);
cudaError_t launch_rscan_rows(int variant, const RScanRowsParams& p, int64_t grid, cudaStream_t s);

// Resident 256-thread blocks per SM for each kernel variant (0 on error).
int occupancy_reduce_contig(int variant);
int occupancy_reduce_rows_warp();
int occupancy_reduce_cols(int variant);
int occupancy_rscan_rows(int variant);

}  // namespace lr
