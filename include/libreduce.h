/*
 * libreduce.h -- C ABI of libreduce on NVIDIA GB300 (sm_103a): fp32
 * reductions (sum, mean, max, min, Euclidean norm; 1D or along one axis) and
 * cumulative sums (forward or reverse, inclusive or exclusive, along any
 * axis), with library or caller-provided scratch.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensor pointers (x, out, y) are DEVICE pointers to memory of the device
 *    that is current on the calling thread (cudaMalloc, the PyTorch caching
 *    allocator, or managed memory).  The caller owns them.  Host pointers are
 *    rejected with LIBREDUCE_ERR_INVALID_ARG before any work is queued.
 *  - Every float* must be 4-byte aligned.  Any 4-byte alignment is accepted;
 *    16-byte aligned buffers take the vectorised (128-bit) paths, and so do
 *    row scans whose x and y sit at the same offset mod 16 bytes (rows of
 *    any length: the float4 items at a row's two edges are masked, and a
 *    masked item's load stays within the 16-byte granule of a row element).
 *  - Arrays are contiguous and row-major.  Sizes are element counts (int64).
 *  - `stream` is a cudaStream_t (NULL means the legacy default stream).  A
 *    call only enqueues work on `stream` and never copies results back; apart
 *    from the one-time workspace set-up described under "Scratch" below, it
 *    never synchronises the host.  The caller keeps the inputs alive and
 *    unmodified until that work completes.  Kernels are launched with
 *    programmatic stream serialization: a call's kernel may begin launching
 *    while the previous kernel on `stream` finishes, but waits for it to
 *    complete (its writes visible) before touching any memory, so stream
 *    order holds as for a plain launch; only launch latency is overlapped.
 *  - Results are deterministic: the same input on the same device gives
 *    bit-identical output on every call.  No floating-point atomics are used;
 *    partial sums are combined in a fixed order.
 *  - Accuracy: each sum or scan output is within 1e-5 * (sum of |x| over its
 *    terms) + 1e-6 of the exact sum, and exact when every partial sum is an
 *    integer of magnitude below 2^24 (max and min are exact; mean and norm as
 *    documented with their op codes).  NaN and Inf propagate as IEEE addition
 *    does.
 *  - Scratch: the library keeps one workspace per device for partial sums,
 *    tickets and error words (17,039,616 bytes) and, once a look-back scan
 *    has run, a second one for look-back node words (2^24 x 8 bytes =
 *    128 MiB).  Each is allocated (cudaMalloc), zeroed (cudaMemset) and
 *    followed by a cudaDeviceSynchronize by the first call on that device that
 *    needs it -- the only time a call synchronises -- so that first call must
 *    not be made inside a stream capture.  Later calls reuse them and
 *    allocate nothing.  Calls that need no scratch (e.g. 1D reductions of at
 *    most 2^18 floats, scans of rows one block per row) never create them.
 *    Because the workspace is shared, calls on one device must not run
 *    concurrently on different streams; calls queued on one stream are always
 *    safe.  The *_ws variants take the scratch from the caller instead and
 *    lift this limit.
 *  - CUDA graphs: after that first call, every call may be captured and the
 *    graph replayed any number of times (tickets are reset on the device, and
 *    the look-back scan takes its launch epoch from a device word that every
 *    launch advances, so a replay never reads an earlier replay's flags).
 *  - Errors: validation happens before any work is queued, and a failed call
 *    queues nothing.  LIBREDUCE_ERR_CUDA means a CUDA runtime call failed; its
 *    code is available from libreduce_last_cuda_error().  Device-side errors
 *    (a bounded wait that ran out) are reported by libreduce_check().
 *
 * Sources (by page):
 *  - "High-Performance Reduction Kernels" (README of a 1D fp32 sum benchmark):
 *    the 1D sum, 'Key design decisions' and 'Optimization: ILP4 accumulator'.
 *  - "Seven-step reduction: 30x from one kernel": warp-shuffle trees, V7.
 *  - POPCORNBENCH trace l1_p47: sum over dim=1 of a contiguous
 *    [128, 4096, 4095] tensor, the [outer, reduce, inner] view.
 *  - POPCORNBENCH trace l1_p91: reverse cumulative sum,
 *    y = cumsum(x.flip(1), 1).flip(1).
 */
#ifndef LIBREDUCE_H_
#define LIBREDUCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported entry points (the library is built with hidden visibility). */
#if defined(__GNUC__)
#define LIBREDUCE_API __attribute__((visibility("default")))
#else
#define LIBREDUCE_API
#endif

/* Same type as cudaStream_t; declared here so callers need no CUDA header. */
typedef struct CUstream_st* libreduce_stream_t;

/* Status codes returned by every entry point. */
#define LIBREDUCE_OK 0
#define LIBREDUCE_ERR_INVALID_ARG 1 /* null pointer with a nonzero extent, negative extent,
                                       misaligned or non-device pointer, bad option */
#define LIBREDUCE_ERR_OVERFLOW 2    /* extent product overflows int64, or exceeds what the
                                       chosen strategy's workspace can hold */
#define LIBREDUCE_ERR_ALIAS 3       /* output overlaps input (the scan is out-of-place only) */
#define LIBREDUCE_ERR_CUDA 4        /* a CUDA runtime call failed (see libreduce_last_cuda_error) */
#define LIBREDUCE_ERR_TIMEOUT 5     /* a bounded device-side wait ran out (from libreduce_check) */
#define LIBREDUCE_ERR_BOUNDS 6      /* debug build only (libreduce_check): a kernel formed an
                                       address outside its call's buffers, or a misaligned
                                       one; the access was skipped (see libreduce_debug_build) */

/*
 * reduce_sum_f32 -- out[0] = sum_{i<n} x[i].
 *
 * The 1D fp32 sum of the "High-Performance Reduction Kernels" README (its
 * benchmark sums n = 1e4 .. 1e9 elements).
 *   x    device, n floats (may be NULL when n == 0)
 *   n    element count, n >= 0; n == 0 writes +0.0f
 *   out  device, 1 float, written once
 * Errors: INVALID_ARG (n < 0, x NULL with n > 0, out NULL, bad pointer),
 *         OVERFLOW (4*n overflows int64), ALIAS (out inside x), CUDA.
 */
LIBREDUCE_API int reduce_sum_f32(const float* x, int64_t n, float* out, libreduce_stream_t stream);

/*
 * reduce_axis_f32 -- out[o*inner + i] = sum_{r<reduce} x[(o*reduce + r)*inner + i].
 *
 * The sum over one axis of a contiguous tensor, viewed as [outer, reduce,
 * inner] (outer = product of the dims before the reduced one, inner = product
 * of the dims after it), as set up in the POPCORNBENCH trace l1_p47 problem
 * statement.  The output is the flat [outer, inner] array; keeping the reduced
 * dim as size 1 is a view for the caller.
 *   x      device, outer*reduce*inner floats
 *   out    device, outer*inner floats, each written once
 *   reduce == 0 writes +0.0f everywhere; outer == 0 or inner == 0 is a no-op.
 * Errors: INVALID_ARG (negative extent, NULL pointer with nonzero size, bad
 *         pointer), OVERFLOW (outer*reduce*inner overflows int64), ALIAS (out
 *         overlaps x), CUDA.
 */
LIBREDUCE_API int reduce_axis_f32(const float* x, int64_t outer, int64_t reduce, int64_t inner, float* out,
                    libreduce_stream_t stream);

/*
 * Other reductions on the same kernels (the "Seven-step reduction" page lists
 * sum, max, the L2 norm and row sums as one pattern):
 *   LIBREDUCE_OP_SUM   sum
 *   LIBREDUCE_OP_MEAN  sum / count (the fp32 sum divided in double, rounded once)
 *   LIBREDUCE_OP_MAX   largest element; NaN if any element is NaN; exact
 *   LIBREDUCE_OP_MIN   smallest element; NaN if any element is NaN; exact
 *   LIBREDUCE_OP_NORM  sqrt(sum of x*x) (correctly rounded square root)
 * An empty reduction gives 0 (sum, norm), NaN (mean), -inf (max), +inf (min).
 * Accuracy: sum as above; mean within (1e-5*sum|x| + 1e-6)/count plus one
 * rounding; norm within 1e-5 * norm + 1e-6.
 *
 * reduce_f32      -- out[0] = op over x[0 .. n-1]             (reduce_sum_f32 is op SUM)
 * reduce_axis_op_f32 -- out[o*inner + i] = op over r of x[(o*reduce + r)*inner + i]
 *                       (reduce_axis_f32 is op SUM)
 * Arguments, layout and errors as reduce_sum_f32 / reduce_axis_f32; an
 * unknown op is INVALID_ARG.
 */
#define LIBREDUCE_OP_SUM 0
#define LIBREDUCE_OP_MEAN 1
#define LIBREDUCE_OP_MAX 2
#define LIBREDUCE_OP_MIN 3
#define LIBREDUCE_OP_NORM 4
LIBREDUCE_API int reduce_f32(const float* x, int64_t n, float* out, int op, libreduce_stream_t stream);
LIBREDUCE_API int reduce_axis_op_f32(const float* x, int64_t outer, int64_t reduce, int64_t inner,
                                     float* out, int op, libreduce_stream_t stream);

/*
 * reverse_cumsum_f32 -- y[i*N + j] = sum_{k=j}^{N-1} x[i*N + k] for every row i.
 *
 * The reverse inclusive cumulative sum along the last dim of a contiguous
 * [rows, N] array, cumsum(x.flip(1), 1).flip(1) in the POPCORNBENCH trace
 * l1_p91 problem statement.  Every output is formed by additions over its own
 * suffix only (no subtraction of prefix sums).
 *   x     device, rows*N floats
 *   y     device, rows*N floats; must not overlap x (out-of-place only)
 *   rows == 0 or N == 0 is a no-op.
 * Rows with few tiles run one block per row; few long rows run a single-pass
 * decoupled look-back scan whose waits are bounded (see libreduce_check).
 * Errors: INVALID_ARG, OVERFLOW (rows*N overflows int64, or a few-row scan
 *         larger than the look-back workspace holds), ALIAS, CUDA.
 */
LIBREDUCE_API int reverse_cumsum_f32(const float* x, int64_t rows, int64_t N, float* y,
                       libreduce_stream_t stream);

/*
 * cumsum_f32 -- cumulative sum along the middle axis of a contiguous
 * [outer, N, inner] array, for every (o, i):
 *   forward (default):              y[o,j,i] = sum_{k <= j} x[o,k,i]
 *   LIBREDUCE_SCAN_REVERSE:         y[o,j,i] = sum_{k >= j} x[o,k,i]
 *   with LIBREDUCE_SCAN_EXCLUSIVE:  the term k == j is left out (k < j, k > j)
 *
 * The generalisation the POPCORNBENCH trace l1_p91 discusses (other scan
 * directions and dims); reverse_cumsum_f32(x, rows, N, y, s) is
 * cumsum_f32(x, rows, N, 1, y, LIBREDUCE_SCAN_REVERSE, s).  inner == 1 scans
 * rows with the row kernels (a forward scan runs as a reverse scan of the
 * mirrored row); inner > 1 scans columns, coalesced across inner (where the
 * (o, column tile) units are too few to fill the GPU, by a single-pass
 * look-back over 256-row x 32-column tiles).  Every
 * output is built from additions over its own terms only (no subtraction),
 * and an exclusive output with no terms is +0.0f.
 *   x     device, outer*N*inner floats
 *   y     device, outer*N*inner floats; must not overlap x
 *   flags LIBREDUCE_SCAN_REVERSE | LIBREDUCE_SCAN_EXCLUSIVE (other bits: INVALID_ARG)
 *   Any zero extent is a no-op.
 * Errors: as reverse_cumsum_f32.
 */
#define LIBREDUCE_SCAN_REVERSE 1u
#define LIBREDUCE_SCAN_EXCLUSIVE 2u
LIBREDUCE_API int cumsum_f32(const float* x, int64_t outer, int64_t N, int64_t inner, float* y,
                             unsigned flags, libreduce_stream_t stream);

/*
 * Workspace variants (the two-call temporary-storage idiom of the CUB
 * DeviceReduce::Sum example on the "Seven-step reduction" page).  They compute
 * exactly what reduce_axis_op_f32 / cumsum_f32 compute, with the same bits,
 * but take their scratch from a caller buffer instead of the library's
 * per-device workspace, so calls with different workspaces may run
 * concurrently on different streams.
 *   ws == NULL:  nothing is queued; *ws_bytes receives the bytes needed: at
 *                least 256 (the header with the call's error word), more when
 *                the call needs partial sums, tickets or look-back flags; 0 for
 *                a call with nothing to compute.  x, y/out and the sizes must be
 *                the ones of the real call (alignment picks the kernels).
 *   ws != NULL:  device memory of the current device, 256-byte aligned, at
 *                least *ws_bytes long (INVALID_ARG if smaller than needed).  The
 *                call clears the parts that must start at zero on `stream`, so
 *                the buffer needs no preparation and may be reused at once.
 *                Its first bytes hold the call's device error word: read it
 *                with libreduce_check_ws(ws, stream).
 * A workspace must not be used by two calls that may overlap on the GPU.
 * Errors: as the plain call; INVALID_ARG for ws_bytes == NULL, a misaligned
 * or too small workspace.
 */
LIBREDUCE_API int reduce_axis_op_ws_f32(const float* x, int64_t outer, int64_t reduce, int64_t inner,
                                        float* out, int op, void* ws, size_t* ws_bytes,
                                        libreduce_stream_t stream);
LIBREDUCE_API int cumsum_ws_f32(const float* x, int64_t outer, int64_t N, int64_t inner, float* y,
                                unsigned flags, void* ws, size_t* ws_bytes, libreduce_stream_t stream);
/* libreduce_check for a workspace call: synchronise `stream`, return and clear
 * the error word in `ws` (LIBREDUCE_OK or LIBREDUCE_ERR_TIMEOUT). */
LIBREDUCE_API int libreduce_check_ws(void* ws, libreduce_stream_t stream);

/*
 * reduce_sum_f32_noalloc -- out[0] = sum_{i<n} x[i], allocating nothing.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory.  reduce_sum_f32 takes its scratch from a
 * workspace the library cudaMallocs on first use; some callers cannot allow
 * that (code inside a custom allocator, or a service whose device memory is
 * capped and every byte budgeted up front).  This call runs the multi-block
 * sum kernel with its scratch (a ticket and up to 16384 partial sums,
 * 64.25 KiB) in a fixed static device array that every GPU loading the
 * library holds until exit.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *   x    device, n floats (may be NULL when n == 0)
 *   n    0 <= n <= 2^36 (16384 blocks of at most 2^22 floats)
 *   out  device, 1 float
 * The result is within the documented tolerance of the exact sum, like
 * reduce_sum_f32's, and the same on every call; the two calls need not give
 * the same bits (reduce_sum_f32 sums arrays of at most 2^18 floats in one
 * thread-block cluster, and this call caps its blocks at 16384).
 * Set-up: the first call on a device (and the first after that device's
 * context was replaced, e.g. by cudaDeviceReset) looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  Every call shares the one array, and the
 * ticket is cleared on the stream before each launch, so calls that overlap
 * on the GPU (different streams, or other threads) race and must be avoided.
 * Errors: INVALID_ARG, OVERFLOW (n > 2^36), ALIAS (out inside x), CUDA.
 */
LIBREDUCE_API int reduce_sum_f32_noalloc(const float* x, int64_t n, float* out, libreduce_stream_t stream);

/*
 * libreduce_check -- synchronise `stream`, then return and clear the current
 * device's error word: LIBREDUCE_OK, or LIBREDUCE_ERR_TIMEOUT if a bounded
 * device-side wait ran out since the last check (the affected outputs are then
 * undefined), or LIBREDUCE_ERR_CUDA if the synchronisation itself failed.
 */
LIBREDUCE_API int libreduce_check(libreduce_stream_t stream);

/* Text for a status code (static storage, never NULL). */
LIBREDUCE_API const char* libreduce_strerror(int status);

/* The cudaError_t of the last CUDA failure seen on this thread (0 if none). */
LIBREDUCE_API int libreduce_last_cuda_error(void);

/* Number of kernels this library has launched in this process (all devices). */
LIBREDUCE_API int64_t libreduce_launch_count(void);

/*
 * Debug build.  The library can also be built with device-side checks
 * (reduction_scan_primitives_gb300.build.build(debug=True) -> libreduce_debug.so,
 * same entry points; no counterpart on the pages): every global access the
 * kernels make through their load/store helpers, their plain output and
 * scratch accesses, and the shared-memory slots of the short-row kernels are
 * checked against the byte ranges of the call's buffers (registered on the
 * call's stream before its launches).  A bad or misaligned access is recorded
 * and skipped -- a load reads zeros, a store is dropped -- never trapped, and
 * libreduce_check / libreduce_check_ws then return LIBREDUCE_ERR_BOUNDS.  The
 * checks are slow, the registration is a host-to-device copy per call (not
 * for stream capture), and concurrent calls on different streams share one
 * registration.
 *   libreduce_debug_build()        1 for the debug build, 0 for the release library
 *   libreduce_debug_bad_address()  the first bad address the last
 *                                  LIBREDUCE_ERR_BOUNDS report found (0: none)
 */
LIBREDUCE_API int libreduce_debug_build(void);
LIBREDUCE_API uint64_t libreduce_debug_bad_address(void);

/*
 * Process-wide dispatch options, for tests and benchmarks.  Not thread-safe
 * against concurrent calls; set them before queuing work.
 *   LIBREDUCE_OPT_SCAN_STRATEGY  0 auto, 1 one block per row, 2 look-back (its fastest
 *                                form), 3 look-back keeping each tile in registers between
 *                                its read and its write (one HBM read, no L2 reread),
 *                                4 reduce-then-scan (tile sums, a scan of the sums, every
 *                                tile scanned again with its carry: three passes),
 *                                5 many short rows (N <= 2048; the automatic choice
 *                                there): chunks of whole rows staged in shared memory,
 *                                each row scanned by a group of 1 to 32 lanes
 *   LIBREDUCE_OPT_AXIS_SPLIT     0 auto, k > 0 forces k slices of the reduce axis
 *                                (inner > 1), or k chunks per row (inner == 1)
 *   LIBREDUCE_OPT_SPIN_LIMIT     0 default, else the look-back wait limit in polls
 *   LIBREDUCE_OPT_STALL_TILE     -1 off, else the look-back tile (in scan order) that
 *                                never publishes its aggregate: a host-chosen fault
 *                                that makes the waits behind it run out, for tests
 * Returns INVALID_ARG for an unknown option or value.
 */
#define LIBREDUCE_OPT_SCAN_STRATEGY 1
#define LIBREDUCE_OPT_AXIS_SPLIT 2
#define LIBREDUCE_OPT_SPIN_LIMIT 3
#define LIBREDUCE_OPT_STALL_TILE 4
/* Launch-shape overrides for tuning sweeps (-1 = automatic):
 *   LIBREDUCE_OPT_CONTIG_VARIANT  loads in flight per thread of the 1D / long-row
 *                                 kernel: 0 -> 4, 1 -> 8, 2 -> 16 (x 16 bytes)
 *   LIBREDUCE_OPT_COLS_VARIANT    inner > 1 kernel: 0..2 scalar columns with 1, 4 or
 *                                 8 warps along the reduce dim; 3..5 the same with
 *                                 float4 columns (needs inner % 4 == 0, aligned x);
 *                                 6, 7 the narrow-row kernel, a block or a warp per plane
 *                                 (inner <= 32 scalar or 128 float4 columns: the
 *                                 automatic choice there); 8 chunks of whole narrow
 *                                 planes (reduce <= 2048, inner <= 256, a plane in
 *                                 24 KB of shared memory), each column reduced as a
 *                                 short row (the automatic choice for planes of at
 *                                 most 768 floats); 9 planes of 2 to 8 columns
 *                                 read flat as segmented class runs (x 16-byte
 *                                 aligned, N >= 2), and of 3 or 5 to 128 columns
 *                                 as column groups (N above the run of 9, 17 or
 *                                 33 rows); the automatic choice from one item
 *                                 of planes per SM on (column groups below 64
 *                                 columns, not on short planes of whole float4
 *                                 rows of 16 columns and more, which a warp per
 *                                 plane takes)
 *   LIBREDUCE_OPT_RSCAN_VARIANT   scan tile: 0 scalar x 4 sub-tiles, 1 float4 x 2,
 *                                 2 float4 x 4 (float4 needs x and y at the same
 *                                 offset mod 16 bytes; any N)
 *   LIBREDUCE_OPT_WAVES           1D sum: blocks = waves x resident blocks (0 = automatic:
 *                                 one wave, or more blocks of 64 Ki floats for long arrays)
 *   LIBREDUCE_OPT_LOOKBACK_LAG    look-back scan: tiles between the read that publishes a
 *                                 tile's sum and the reread that writes it (0 = automatic)
 *   LIBREDUCE_OPT_SCAN_COLS_VARIANT  scan along a strided axis (inner > 1), block shape:
 *                                 0 scalar columns, 2 warps across x 4 down the axis;
 *                                 1 float4 columns, 2 x 4; 2 float4 columns, 1 x 8;
 *                                 3, 4 the narrow-row scan, tiles in shared memory or a
 *                                 warp per (plane, segment) (inner <= 32 scalar or 128
 *                                 float4 columns: the automatic choice there);
 *                                 5 the single-pass look-back over 256-row x 32-column
 *                                 tiles (the automatic choice where one block per
 *                                 (o, column tile) cannot fill the GPU; falls back to
 *                                 the automatic choice when its tiles exceed 262144);
 *                                 6 chunks of whole narrow planes (N <= 2048,
 *                                 inner <= 256, a plane in 24 KB of shared memory),
 *                                 each column scanned as a short row (the automatic
 *                                 choice wherever a plane fits); 7 planes of 2 or 4
 *                                 columns read flat as rows (x and y at the same
 *                                 offset mod 16 bytes), each column a class of
 *                                 every 2nd or 4th element, by the row kernels
 *                                 (the automatic choice for 2-column planes of at
 *                                 least 4096 floats, after forms 8 and 9); 8 planes
 *                                 of 2 to 8, 9, 10, 12 or 14 columns read flat as
 *                                 segmented class runs (x and y 16-byte aligned,
 *                                 N >= 2), and of 6 to 128 columns as column
 *                                 groups where the planes are longer than their
 *                                 runs (a float4, float2 or float of adjacent
 *                                 columns per thread over runs of 9, 17 or 33
 *                                 rows); the automatic choice from one item per
 *                                 SM on (column groups of 64 or 128 columns only
 *                                 below 256 rows), an item being one plane or
 *                                 several short planes (up to 8 tiles of them
 *                                 for column groups); 9 the same tiles with a
 *                                 plane's tiles spread over blocks and their carries
 *                                 from a look-back (the automatic choice for fewer
 *                                 items than SMs when planes hold two tiles or more;
 *                                 column groups for 7 to 128 columns, but 64 and 128)
 *                                 (float4 columns need inner % 4 == 0 and aligned x, y) */
#define LIBREDUCE_OPT_CONTIG_VARIANT 5
#define LIBREDUCE_OPT_COLS_VARIANT 6
#define LIBREDUCE_OPT_RSCAN_VARIANT 7
#define LIBREDUCE_OPT_WAVES 8
#define LIBREDUCE_OPT_LOOKBACK_LAG 9
#define LIBREDUCE_OPT_SCAN_COLS_VARIANT 10
/* LIBREDUCE_OPT_ROWS_FORM  reductions along rows of at most 2048 elements (inner == 1):
 *                          0 automatic (2 up to 128 elements, else 1), 1 one warp per
 *                          row, 2 chunks of whole rows staged in shared memory, a
 *                          group of 1 to 32 lanes per row */
#define LIBREDUCE_OPT_ROWS_FORM 11
LIBREDUCE_API int libreduce_set_option(int option, int64_t value);

#ifdef __cplusplus
}
#endif

#endif /* LIBREDUCE_H_ */
