// lr_api.cu -- the C ABI of libreduce: argument validation, strategy choice,
// workspace management and kernel launches.  See include/libreduce.h for the
// contract of each entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstddef>
#include <cstring>
#include <mutex>

#include "libreduce.h"
#include "lr_internal.h"

namespace lr {

#ifdef LR_DEBUG
__device__ LrDebug g_lr_debug;  // the debug build's registered ranges and findings
#endif

namespace {

// ---------------------------------------------------------------------------
// Process state.
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxTickets = 1 << 16;       // integer tickets (per row / column tile)
constexpr int64_t kMaxPartials = 1 << 22;      // fp32 partial sums (16 MiB)
constexpr size_t kHeaderBytes = 256;           // error word, abort word, {ticket counter, epoch}
// Look-back node words (allocated on the first look-back of a device, 128 MB):
// a row look-back takes 2 words per tile, a column look-back 2 per tile and
// column.
constexpr int64_t kLookbackWords = int64_t(1) << 24;
constexpr int64_t kMaxLookbackTiles = kLookbackWords / 2;  // row look-back tiles per launch
constexpr size_t kWorkspaceBytes =
    kHeaderBytes + sizeof(unsigned) * kMaxTickets + sizeof(float) * kMaxPartials;

struct DeviceState {
  bool ready = false;
  int sm_count = 0;
  int occ_contig[kNumContigVariants][kNumReduceOps] = {};
  int occ_rows_warp[kNumReduceOps] = {};
  int occ_cols[kNumColsVariants][kNumReduceOps] = {};
  int occ_rscan[kNumRScanVariants] = {};
  // Workspace (allocated by the first call that needs it).
  char* ws = nullptr;
  unsigned* err_word = nullptr;
  unsigned* tickets = nullptr;
  float* partials = nullptr;
  // Look-back region (allocated by the first look-back scan on the device).
  unsigned long long* node_val = nullptr;
  int occ_lookback[kNumLookbackVariants] = {};
  int occ_scan_cols[kNumScanColsVariants] = {};
  int occ_narrow[2][kNumReduceOps] = {};  // [vec4][op]
  int occ_scan_narrow[2] = {};            // [vec4]
  int occ_scan_narrow_warp[2] = {};       // [vec4]
  int occ_scan_cols_lb = 0;
  int occ_rscan_short = 0;
  int occ_rscan_period[3] = {};     // float4 block per row, period 1, 2, 4
  int occ_lookback_period[3] = {};  // L2 look-back, period 1, 2, 4
  int occ_planes[kPlanesMaxScanP - 1][2] = {};  // narrow planes read flat: [P - 2][scan]
  int occ_planes_lb[kPlanesMaxP - 1] = {};  // the same, look-back form: [P - 2]
  int occ_planes_cg[kPlanesCgInstances] = {};  // scans as column groups, by instance
  int occ_planes_cg_reduce[kPlanesCgInstances] = {};  // reductions as column groups
  int occ_planes_cg_lb[kPlanesCgInstances] = {};      // few long planes as column groups
};

// Index of a period (1, 2, 4) in the per-period tables.
int period_slot(int period) { return period == 4 ? 2 : period == 2 ? 1 : 0; }

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<int64_t> g_launches{0};
std::atomic<int64_t> g_opt_scan_strategy{0};
std::atomic<int64_t> g_opt_axis_split{0};
std::atomic<int64_t> g_opt_spin_limit{0};
std::atomic<int64_t> g_opt_stall_tile{-1};
std::atomic<int64_t> g_opt_contig_variant{-1};
std::atomic<int64_t> g_opt_cols_variant{-1};
std::atomic<int64_t> g_opt_rscan_variant{-1};
std::atomic<int64_t> g_opt_scan_cols_variant{-1};
std::atomic<int64_t> g_opt_rows_form{0};
std::atomic<int64_t> g_opt_waves{0};
std::atomic<int64_t> g_opt_lookback_lag{0};
thread_local int t_last_cuda_error = 0;
// Debug builds: the current call's input and output byte ranges (set by the
// entry point, registered with the scratch when the call acquires it), and
// the first bad address the last check found.
thread_local const void* t_dbg_buf[2] = {nullptr, nullptr};
thread_local size_t t_dbg_bytes[2] = {0, 0};
std::atomic<unsigned long long> g_dbg_last_bad{0};
void dbg_call_buffers(const void* in, size_t in_bytes, const void* out, size_t out_bytes) {
  t_dbg_buf[0] = in;
  t_dbg_bytes[0] = in_bytes;
  t_dbg_buf[1] = out;
  t_dbg_bytes[1] = out_bytes;
}

int fail_cuda(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return LIBREDUCE_ERR_CUDA;
}

// Query the current device and fill its cached properties.
int device_state(DeviceState** out, int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return LIBREDUCE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail_cuda(e);
    for (int op = 0; op < kNumReduceOps; ++op) {
      for (int v = 0; v < kNumContigVariants; ++v)
        st.occ_contig[v][op] = std::max(1, occupancy_reduce_contig(v, op));
      st.occ_rows_warp[op] = std::max(1, occupancy_reduce_rows_warp(op));
      for (int v = 0; v < kNumColsVariants; ++v)
        st.occ_cols[v][op] = std::max(1, occupancy_reduce_cols(v, op));
    }
    for (int v = 0; v < kNumRScanVariants; ++v) st.occ_rscan[v] = std::max(1, occupancy_rscan_rows(v));
    for (int v = 0; v < kNumLookbackVariants; ++v)
      st.occ_lookback[v] = std::max(1, occupancy_rscan_lookback(v));
    for (int v = 0; v < kNumScanColsVariants; ++v)
      st.occ_scan_cols[v] = std::max(1, occupancy_scan_cols(v));
    for (int v4 = 0; v4 < 2; ++v4) {
      for (int op = 0; op < kNumReduceOps; ++op)
        st.occ_narrow[v4][op] = std::max(1, occupancy_reduce_narrow(v4 ? 4 : 1, op));
      st.occ_scan_narrow[v4] = std::max(1, occupancy_scan_narrow(v4 ? 4 : 1));
      st.occ_scan_narrow_warp[v4] = std::max(1, occupancy_scan_narrow_warp(v4 ? 4 : 1));
    }
    st.occ_scan_cols_lb = std::max(1, occupancy_scan_cols_lookback());
    for (int pi = 0; pi < 3; ++pi) {
      st.occ_rscan_period[pi] = std::max(1, occupancy_rscan_rows_period(1 << pi));
      st.occ_lookback_period[pi] = std::max(1, occupancy_rscan_lookback_period(1 << pi));
    }
    st.occ_rscan_short = std::max(1, occupancy_rscan_short());
    for (int pi = 0; pi < kPlanesMaxScanP - 1; ++pi) {
      const int P = pi + 2;
      if (planes_scan_columns(P)) st.occ_planes[pi][1] = std::max(1, occupancy_planes(P, true));
      if (P > kPlanesMaxP) continue;
      st.occ_planes[pi][0] = std::max(1, occupancy_planes(P, false));
      st.occ_planes_lb[pi] = std::max(1, occupancy_planes_lookback(P));
    }
    for (int ci = 0; ci < kPlanesCgInstances; ++ci) {
      st.occ_planes_cg[ci] = std::max(1, occupancy_planes_cg(ci));
      st.occ_planes_cg_reduce[ci] = std::max(1, occupancy_planes_cg_reduce(ci));
      st.occ_planes_cg_lb[ci] = std::max(1, occupancy_planes_cg_lookback(ci));
    }
    cudaGetLastError();  // occupancy queries leave no error behind
    st.ready = true;
  }
  *out = &st;
  if (dev_out) *dev_out = dev;
  return LIBREDUCE_OK;
}

// Allocate and zero the device workspace once per device.
int ensure_workspace(DeviceState* st) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (st->ws) return LIBREDUCE_OK;
  void* p = nullptr;
  cudaError_t e = cudaMalloc(&p, kWorkspaceBytes);
  if (e != cudaSuccess) return fail_cuda(e);
  e = cudaMemset(p, 0, kWorkspaceBytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(p);
    return fail_cuda(e);
  }
  char* base = static_cast<char*>(p);
  st->ws = base;
  st->err_word = reinterpret_cast<unsigned*>(base);
  st->tickets = reinterpret_cast<unsigned*>(base + kHeaderBytes);
  st->partials = reinterpret_cast<float*>(base + kHeaderBytes + sizeof(unsigned) * kMaxTickets);
  return LIBREDUCE_OK;
}

// Allocate the look-back flags once per device.  Their epochs (a device word
// in the header, advanced by every look-back launch) make stale contents
// harmless, but they start zeroed (epoch 0 is never used).
int ensure_lookback(DeviceState* st) {
  int rc = ensure_workspace(st);
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  if (st->node_val) return LIBREDUCE_OK;
  const size_t nodes = (size_t)kLookbackWords;
  const size_t bytes = nodes * sizeof(unsigned long long);
  void* p = nullptr;
  cudaError_t e = cudaMalloc(&p, bytes);
  if (e != cudaSuccess) return fail_cuda(e);
  e = cudaMemset(p, 0, bytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(p);
    return fail_cuda(e);
  }
  st->node_val = static_cast<unsigned long long*>(p);
  return LIBREDUCE_OK;
}

// ---------------------------------------------------------------------------
// Validation.
// ---------------------------------------------------------------------------
using GetAddressRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);

GetAddressRangeFn address_range_fn() {
  static GetAddressRangeFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      f = nullptr;
    }
    return reinterpret_cast<GetAddressRangeFn>(f);
  }();
  return fn;
}

// `p` must be device (or managed) memory of device `dev`, 4-byte aligned, and
// [p, p + bytes) must lie inside one allocation.  This keeps a wrong size or a
// host pointer from ever reaching a kernel.
int check_buffer(const void* p, size_t bytes, int dev) {
  if (p == nullptr) return LIBREDUCE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(p) & 3u) return LIBREDUCE_ERR_INVALID_ARG;
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return LIBREDUCE_ERR_INVALID_ARG;
  }
  if (a.type == cudaMemoryTypeDevice) {
    if (a.device != dev) return LIBREDUCE_ERR_INVALID_ARG;
  } else if (a.type != cudaMemoryTypeManaged) {
    return LIBREDUCE_ERR_INVALID_ARG;
  }
  GetAddressRangeFn fn = address_range_fn();
  if (fn) {
    CUdeviceptr base = 0;
    size_t size = 0;
    if (fn(&base, &size, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS) return LIBREDUCE_ERR_INVALID_ARG;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    if (lo < base || bytes > size || lo - base > size - bytes) return LIBREDUCE_ERR_INVALID_ARG;
  }
  return LIBREDUCE_OK;
}

bool mul_overflows(int64_t a, int64_t b, int64_t* r) {
  return __builtin_mul_overflow(a, b, r);
}

bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes) {
  if (abytes == 0 || bbytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bbytes && b0 < a0 + abytes;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t m) { return ceil_div(a, m) * m; }

int launched(cudaError_t e) {
  if (e != cudaSuccess) return fail_cuda(e);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return LIBREDUCE_OK;
}

// ---------------------------------------------------------------------------
// Strategies.
// ---------------------------------------------------------------------------
constexpr int64_t kMinChunk = 8192;         // floats per block, lower bound
constexpr int64_t kClusterSlice = 16384;    // floats per CTA of a short 1D array (one cluster)
constexpr int64_t kPeriodRowsMin = 4096;    // planes of 2 or 4 columns from this many floats: flat rows
constexpr int64_t kTargetChunk = 65536;     // floats per block of a long 1D sum (256 KiB)
constexpr int64_t kRowsWarpMaxLen = 2048;   // rows up to this length: one warp per row
constexpr int64_t kShortReduceMax = 128;    // rows up to this length: staged chunks (automatic choice;
                                            // measured 0.75 against 0.21 at N = 32, 0.54 against
                                            // 0.31 at 100, and behind one warp per row from 256)
// Short-row plans (short_form): rows up to these lengths (odd lengths: *Odd)
// take one lane each.  A lane walks its row with sequential additions, so
// an output can end a chain of N - 1 roundings; at most 158 keeps the
// worst case, 158 * 2^-24 * sum|x| (to first order), inside the tolerance
// 1e-5 * sum|x| for any data.  (Odd rows up to 255 scanned 0.70-0.81 walked
// against 0.64 in lane groups; a walk with a carry folded every 16 elements,
// which would bound the chain, cost 15-20% at every length.)
constexpr int64_t kShortScanSolo = 64;
constexpr int64_t kShortScanSoloOdd = 159;
constexpr int64_t kShortReduceSolo = 64;
constexpr int64_t kShortReduceSoloOdd = kShortReduceMax;

int contig_variant() {
  const int64_t v = g_opt_contig_variant.load();
  return (v >= 0 && v < kNumContigVariants) ? (int)v : kContigU16;
}

// ---------------------------------------------------------------------------
// Scratch.  Every strategy first states what it needs; a provider then hands
// it out from the library's per-device workspace or from a caller buffer
// (the *_ws entry points).  The plan never depends on the provider, so both
// give bit-identical results.
// ---------------------------------------------------------------------------
struct Need {
  int64_t tickets = 0;   // u32, zero on entry
  int64_t partials = 0;  // f32
  int64_t nodes = 0;     // u64 look-back words, zero (or stale-epoch) on entry
  bool header = false;   // error / abort / ticket-counter words
};

struct Scratch {
  unsigned* header = nullptr;
  unsigned* tickets = nullptr;
  float* partials = nullptr;
  unsigned long long* nodes = nullptr;
};

struct Provider {
  DeviceState* st = nullptr;
  char* ws = nullptr;        // caller workspace, or null for the library's own
  size_t ws_bytes = 0;
  size_t* query = nullptr;   // size query: store the bytes needed, launch nothing
};

constexpr int kQueried = -1;  // internal: a size query was answered

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

// Caller-workspace layout: [header 256 B][tickets][partials][nodes], each part
// 256-byte aligned.
void ws_layout(const Need& n, size_t* off_t, size_t* off_p, size_t* off_n, size_t* total) {
  *off_t = kHeaderBytes;
  *off_p = *off_t + align256(sizeof(unsigned) * (size_t)n.tickets);
  *off_n = *off_p + align256(sizeof(float) * (size_t)n.partials);
  *total = *off_n + align256(sizeof(unsigned long long) * (size_t)n.nodes);
}

// Debug builds: register the call's buffers and every scratch region it may
// touch, on the call's stream, before its launches.
int register_call(const Provider& pv, cudaStream_t s) {
#ifdef LR_DEBUG
  const void* p[kDbgRanges] = {t_dbg_buf[0], t_dbg_buf[1], nullptr, nullptr, nullptr, nullptr};
  size_t b[kDbgRanges] = {t_dbg_bytes[0], t_dbg_bytes[1], 0, 0, 0, 0};
  if (pv.ws) {
    p[2] = pv.ws;
    b[2] = pv.ws_bytes;
  } else if (pv.st) {
    p[2] = pv.st->ws;
    b[2] = pv.st->ws ? kWorkspaceBytes : 0;
    p[3] = pv.st->node_val;
    b[3] = pv.st->node_val ? sizeof(unsigned long long) * (size_t)kLookbackWords : 0;
  }
  const cudaError_t e = dbg_register_ranges(s, p, b, kDbgRanges);
  if (e != cudaSuccess) return fail_cuda(e);
#else
  (void)pv;
  (void)s;
#endif
  return LIBREDUCE_OK;
}

int acquire_impl(const Provider& pv, const Need& need, Scratch* sc, cudaStream_t s) {
  const bool any = need.tickets || need.partials || need.nodes || need.header;
  if (pv.query) {
    // A caller workspace always holds at least the header (its error word).
    size_t a, b, c, total = 0;
    ws_layout(need, &a, &b, &c, &total);
    *pv.query = total;
    return kQueried;
  }
  if (!pv.ws) {
    if (!any) return LIBREDUCE_OK;
    DeviceState* st = pv.st;
    int rc = need.nodes ? ensure_lookback(st) : ensure_workspace(st);
    if (rc) return rc;
    sc->header = st->err_word;
    sc->tickets = st->tickets;
    sc->partials = st->partials;
    sc->nodes = st->node_val;
    return LIBREDUCE_OK;
  }
  size_t off_t, off_p, off_n, total;
  ws_layout(need, &off_t, &off_p, &off_n, &total);
  if (total > pv.ws_bytes) return LIBREDUCE_ERR_INVALID_ARG;  // workspace too small
  // A caller workspace holds anything on entry: clear what must start at zero.
  cudaError_t e = cudaMemsetAsync(pv.ws, 0, off_p, s);
  if (e == cudaSuccess && need.nodes)
    e = cudaMemsetAsync(pv.ws + off_n, 0, sizeof(unsigned long long) * (size_t)need.nodes, s);
  if (e != cudaSuccess) return fail_cuda(e);
  sc->header = reinterpret_cast<unsigned*>(pv.ws);
  sc->tickets = reinterpret_cast<unsigned*>(pv.ws + off_t);
  sc->partials = reinterpret_cast<float*>(pv.ws + off_p);
  sc->nodes = reinterpret_cast<unsigned long long*>(pv.ws + off_n);
  return LIBREDUCE_OK;
}

// Every strategy takes its scratch here before launching: the scratch first
// (so its ranges exist), then, in debug builds, the call's registration.
int acquire(const Provider& pv, const Need& need, Scratch* sc, cudaStream_t s) {
  const int rc = acquire_impl(pv, need, sc, s);
  if (rc || pv.query) return rc;
  return register_call(pv, s);
}

// Reduction of `segments` contiguous segments of seg_len floats each.
int run_contig(const Provider& pv, const float* x, int64_t segments, int64_t seg_len, float* out,
               int op, int epi, cudaStream_t s) {
  DeviceState* st = pv.st;
  const int variant = op == kOpSum ? contig_variant() : kContigU16;
  const int64_t slots = (int64_t)st->sm_count * st->occ_contig[variant][op];
  const int64_t waves = g_opt_waves.load();
  int64_t chunks = 1;
  const int64_t forced = g_opt_axis_split.load();
  if (segments == 1 && seg_len > kClusterSlice && seg_len <= kClusterMaxN && forced <= 0 && waves <= 0 &&
      g_opt_contig_variant.load() < 0) {
    // A short array: one cluster of CTAs, about kClusterSlice floats each
    // (all of a CTA's loads in one round trip), combined in distributed
    // shared memory: one launch, no scratch, no ticket.  Up to kClusterSlice
    // floats one plain block does it (below, chunks == 1), which launches
    // faster than a cluster (measured per launch in a graph: 1.95 against
    // 2.7 us at 1e4; at 1e5 the cluster takes 2.95 against 3.54 us for 12
    // blocks and a ticket).
    Scratch sc;
    int rc = acquire(pv, Need{}, &sc, s);
    if (rc) return rc;
    int64_t ctas = std::min<int64_t>(kClusterMaxCtas, std::max<int64_t>(1, ceil_div(seg_len, kClusterSlice)));
    const int64_t len = round_up(ceil_div(seg_len, ctas), 4);
    ctas = ceil_div(seg_len, len);
    ContigParams p{x, seg_len, len, (int32_t)ctas, out, nullptr, nullptr, epi};
    return launched(launch_reduce_cluster(op, p, (int)ctas, s));
  }
  if (forced > 0) {
    chunks = std::min<int64_t>(forced, ceil_div(seg_len, 4));
  } else if (segments == 1) {
    // One long array: a whole number of waves of resident blocks, each block
    // about kTargetChunk floats.  A partial last wave would cost a whole
    // block's duration for a few blocks (measured: 1526 blocks at 1e8 take 16%
    // longer than 1520).
    const int64_t w = waves > 0 ? waves
                                : std::max<int64_t>(1, (seg_len + kTargetChunk * slots / 2) /
                                                           (kTargetChunk * slots));
    chunks = w * slots;
    chunks = std::min(chunks, std::max<int64_t>(1, seg_len / kMinChunk));
    if (seg_len <= kClusterSlice && waves <= 0) chunks = 1;  // one block, one round trip, no ticket
  } else if (segments < 4 * slots) {
    // Too few rows to fill the GPU: cut each into chunks.
    chunks = ceil_div(4 * slots, segments);
    chunks = std::min(chunks, std::max<int64_t>(1, seg_len / kMinChunk));
  }
  int64_t chunk_len = round_up(ceil_div(seg_len, chunks), 4);
  chunks = ceil_div(seg_len, chunk_len);
  if (chunks > 1 && (segments > kMaxTickets || segments * chunks > kMaxPartials)) {
    chunks = 1;
    chunk_len = round_up(seg_len, 4);
  }
  const int64_t grid = segments * chunks;
  if (grid > INT32_MAX) return LIBREDUCE_ERR_OVERFLOW;
  Need need;
  if (chunks > 1) {
    need.tickets = segments;
    need.partials = segments * chunks;
  }
  Scratch sc;
  int rc = acquire(pv, need, &sc, s);
  if (rc) return rc;
  ContigParams p{x, seg_len, chunk_len, (int32_t)chunks, out, sc.partials, sc.tickets, epi};
  return launched(launch_reduce_contig(variant, op, p, grid, s));
}

int run_rows_short(const Provider& pv, const float* x, int64_t rows, int64_t N, float* out, int op, int epi,
                   cudaStream_t s);
// Reductions of narrow planes by the short-row kernels (defined with them
// below); kNoPlanes when the planes do not fit a chunk.
constexpr int64_t kDefaultSpinLimit = 1 << 20;  // polls (with short sleeps): well under a second
constexpr int kColLbNoFit = -2;  // distinct from kQueried
constexpr int kNoPlanes = -3;  // distinct from kQueried and kColLbNoFit
constexpr int64_t kShortPlaneInnerMax = 256;  // widest plane the short-row kernels take
constexpr int64_t kShortPlaneAutoInnerMax = 64;  // widest plane the automatic choice gives them
int try_reduce_short_planes(const Provider& pv, const float* x, int64_t outer, int64_t N, int64_t inner,
                            float* out, int op, int epi, bool forced, cudaStream_t s);

int run_rows_warp(const Provider& pv, const float* x, int64_t rows, int64_t len, float* out, int op,
                  int epi, cudaStream_t s) {
  DeviceState* st = pv.st;
  const int64_t slots = (int64_t)st->sm_count * st->occ_rows_warp[op];
  const int64_t grid = std::max<int64_t>(1, std::min(ceil_div(rows, kThreads / 32), 8 * slots));
  Scratch sc;
  int rc = acquire(pv, Need{}, &sc, s);
  if (rc) return rc;
  RowsWarpParams p{x, rows, len, out, epi};
  return launched(launch_reduce_rows_warp(op, p, grid, s));
}

// Narrow rows: at most 256 scalar or 128 float4 columns (VEC = 4 when inner
// % 4 == 0 and x, y are 16-byte aligned).  Beyond that the wide kernels keep
// every lane busy (and reach the copy bandwidth on 16-byte aligned rows).
bool narrow_rows(const float* x, const float* y, int64_t inner, int* vec) {
  const bool vec4 = (inner % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) &&
                    ((reinterpret_cast<uintptr_t>(y) & 15u) == 0);
  *vec = vec4 ? 4 : 1;
  return inner > 1 && inner <= (vec4 ? 128 : 256);
}

// A warp per plane pays when the planes are many and small: a block per plane
// would spend its time starting up, and there are enough planes to fill the
// GPU with warps (measured on [100000, 100, 3]: 46% against 6% of copy
// bandwidth; on [1024, 8192, 64] the block form is ahead, 99% against 81%).
bool narrow_warp_reduce(const DeviceState* st, int64_t outer, int64_t reduce, int64_t inner, int vec) {
  return inner <= 32 * vec && outer >= (int64_t)st->sm_count * 32 && reduce * inner <= 64 * 1024;
}

// Axis reduction over narrow rows: one block per (o, slice); when outer alone
// cannot fill the GPU the reduce axis is sliced so the grid is one full wave
// (as run_cols does), each slice at least one step of U = 8 rows per row
// group; the last block of o combines the slices.
int run_narrow(const Provider& pv, const float* x, int64_t outer, int64_t reduce, int64_t inner,
               float* out, int op, int epi, int vec, int64_t forced_splits, cudaStream_t s) {
  DeviceState* st = pv.st;
  const int64_t slots = (int64_t)st->sm_count * st->occ_narrow[vec == 4][op];
  const int64_t groups = kThreads / (inner / vec);
  int64_t splits = 1;
  if (forced_splits > 0) {
    splits = std::min(forced_splits, reduce);
  } else if (outer < slots) {
    splits = std::max<int64_t>(1, slots / outer);
    splits = std::min(splits, std::max<int64_t>(1, reduce / (8 * groups)));
  }
  if (splits > 1) {  // the slices must fit the tickets and partials
    const int64_t cap = outer > kMaxTickets ? 1 : kMaxPartials / (outer * inner);
    splits = cap < 2 ? 1 : std::min(splits, cap);
  }
  int64_t rows_per_split = ceil_div(reduce, splits);
  splits = ceil_div(reduce, rows_per_split);
  int64_t grid = 0;
  if (mul_overflows(outer, splits, &grid) || grid > INT32_MAX) return LIBREDUCE_ERR_OVERFLOW;
  Need need;
  if (splits > 1) {
    need.tickets = outer;
    need.partials = outer * splits * inner;
  }
  Scratch sc;
  int rc = acquire(pv, need, &sc, s);
  if (rc) return rc;
  NarrowParams p{x, outer, reduce, inner, splits, rows_per_split, out, sc.partials, inner,
                 sc.tickets, epi, 0};
  return launched(launch_reduce_narrow(vec, op, p, grid, s));
}

// Narrow planes read flat as segmented class runs (lr_planes.cuh): 2-8
// columns, and for scans also 9, 10, 12 and 14; scans of every other column
// count up to 128 as column groups.  Planes per item and items,
// or false when the shape does not fit (planes of one row).  Short planes go k >= 2 to a tile (the item's
// start is rounded down to planes_align floats), planes no longer than a
// thread's run with several boundaries in a run; longer ones one to an item.
struct PlaneRunPlan {
  int64_t k = 1, items = 0;
  unsigned long long magic = 0;
  bool multi = false;  // planes no longer than a thread's run: several boundaries in a run
  bool cg = false;     // column groups (k_planes_cg)
};
bool plane_run_plan(int64_t outer, int64_t N, int64_t inner, PlaneRunPlan* pl, bool scan, bool allow_cg = true) {
  int64_t L = 0;
  if (inner < 2 || outer <= 0 || N < 2 || mul_overflows(N, inner, &L)) return false;
  if (allow_cg && inner <= kPlanesCgMaxP && (scan ? planes_cg_scan((int)inner) : planes_cg_reduce((int)inner)) &&
      N > planes_cg_run_rows((int)inner)) {
    // Column groups: tiles of whole rows, boundaries in rows.  Items of
    // several planes may span up to 8 tiles (while that leaves 2048 items
    // or more), so that only an item's last tile runs part full: short
    // planes one to a tile would leave up to half of it idle.
    const int64_t TR = planes_cg_tile_rows((int)inner);
    int64_t rows = 0;
    const int64_t per =
        mul_overflows(outer, N, &rows) ? 1 : std::max<int64_t>(1, std::min<int64_t>(8, ceil_div(rows, TR) / 2048));
    const int64_t k = TR * per / N;
    pl->k = k >= 2 ? k : 1;
    pl->items = ceil_div(outer, pl->k);
    pl->magic = pl->k >= 2 ? ((1ull << 32) + (unsigned long long)N - 1) / (unsigned long long)N : 0;
    pl->multi = false;
    pl->cg = true;
    return true;
  }
  if (inner > kPlanesMaxScanP || (!scan && inner > kPlanesMaxP) || !planes_scan_columns((int)inner)) return false;
  pl->cg = false;
  const int64_t align = planes_align((int)inner);
  const int64_t k = (planes_tile_len((int)inner) - align + 1) / L;
  pl->k = k >= 2 ? k : 1;
  pl->items = ceil_div(outer, pl->k);
  pl->magic = pl->k >= 2 ? ((1ull << 32) + (unsigned long long)L - 1) / (unsigned long long)L : 0;
  pl->multi = L <= planes_run_len((int)inner);
  return true;
}
// The automatic choice takes the flat runs when there is at least one item
// per SM.  A block streams about 33 GB/s of a scan, so from ~150 items on the
// runs pass the forms that split a plane across blocks (fractions of copy
// bandwidth, runs against the automatic choice before them: [512, 3000, 3]
// 0.93 / 0.27, [400, 10000, 3] 0.80 / 0.30, [300, 5000, 4] 0.80 / 0.65,
// [200, 50000, 4] 0.83 / 0.56, [100, 20000, 2] 0.49 / 0.31; sums [512, 3000,
// 3] 0.69 / 0.37, [300, 5000, 4] 0.64 / 0.38); with only tens of planes a
// block per plane leaves most SMs idle.
// Eight columns (two float4s a row) keep the narrow kernels for planes of a
// tile or more and for reductions, which those read as whole float4 rows
// (fractions, runs against them: scans [1000, 10000, 8] 0.72 / 0.83, sums
// [100000, 100, 8] 0.57 / 0.60; short-plane scans [100000, 100, 8] 0.89 /
// 0.54 take the runs).
// Planes no longer than a thread's run take the runs too: scans [500000,
// 7, 3] 0.87 against 0.53, [2e6, 8, 2] 0.88 against 0.64, [1e6, 4, 8] 0.84
// against 0.62; sums [500000, 7, 3] 0.74 against 0.39, [2e6, 8, 2] 0.81
// against 0.63, [1e6, 3, 6] 0.52 against 0.41.  Scans as column groups
// (11 to 128 columns, and 16 and 32) against the best other form: [58181,
// 100, 11] 0.89 / 0.50, [4923, 1000, 13] 0.84 / 0.41, [40000, 100, 16] 0.92
// / 0.41, [3555, 1000, 18] 0.89 / 0.43, [26666, 100, 24] 0.92 / 0.52,
// [2064, 1000, 31] 0.87 / 0.63, [1333, 1000, 48] 0.87 / 0.73, [10000, 100,
// 64] 0.88 / 0.82, [6400, 100, 100] 0.85 / 0.70, [640, 1000, 100] 0.81 /
// 0.69, [5000, 100, 128] 0.89 / 0.82.  Planes of 64 or 128 columns (whole
// 32-column tiles for the other forms) and 256 rows or more stay with
// those ([3906, 256, 64] 0.88 / 0.91, [1000, 1000, 64] 0.82 / 0.89,
// [1953, 256, 128] 0.85 / 0.97).  Reductions as column groups (9 to 63
// columns): [7111, 1000, 9] 0.91 / 0.63, [5818, 1000, 11] 0.90 / 0.45,
// [3764, 1000, 17] 0.91 / 0.74, [71111, 100, 9] 0.85 / 0.81, [37647, 100,
// 17] 0.87 / 0.62; a warp per plane stays ahead on short planes of whole
// float4 rows ([26666, 100, 24] 0.98 / 0.85, [20000, 100, 32] 1.01 /
// 0.90), and the narrow and short-row forms from 64 columns on ([640,
// 1000, 100] 0.93 / 0.74, [500, 1000, 128] 0.92 / 0.67).
bool plane_runs_fill(const DeviceState* st, const PlaneRunPlan& pl, int64_t outer, int64_t N, int64_t inner,
                     bool scan) {
  if (!pl.cg && inner == 8 && (!scan || pl.k < 2)) return false;
  if (pl.cg && scan && inner % 32 == 0 && inner >= 64 && N >= 256) return false;
  if (pl.cg && !scan &&
      (inner >= 64 || (inner >= 16 && inner % 4 == 0 && narrow_warp_reduce(st, outer, N, inner, 4))))
    return false;
  return pl.items >= st->sm_count;
}
// Fewer items than SMs: the look-back form, whose blocks take single tiles,
// when the planes hold at least two tiles each (measured in the plane-run
// tests; below that the items' blocks are few and short either way).
// Only with runs of 36 floats (2, 3, 4, 6 columns): the shorter tiles of 5,
// 7 and 8 columns leave one block per 10-12 KB tile too little to do
// ([1, 3e7, 5] 0.48, [2, 2e7, 8] 0.39 of copy bandwidth).
bool plane_runs_split(const DeviceState* st, const PlaneRunPlan& pl, int64_t N, int64_t inner) {
  return planes_run_len((int)inner) == 36 && pl.items < st->sm_count && N * inner >= 2 * planes_tile_len((int)inner);
}
int run_planes(const Provider& pv, const PlaneRunPlan& pl, const float* x, int64_t outer, int64_t N,
               int64_t inner, float* y, int flags, bool scan, int op, cudaStream_t s) {
  DeviceState* st = pv.st;
  Need need;
  need.header = true;  // the error word (a copy that never lands)
  Scratch sc;
  const int rc = acquire(pv, need, &sc, s);
  if (rc) return rc;
  const int ci = pl.cg ? cg_instance((int)inner) : 0;
  const int occ = pl.cg ? (scan ? st->occ_planes_cg[ci] : st->occ_planes_cg_reduce[ci])
                        : st->occ_planes[inner - 2][scan ? 1 : 0];
  const int64_t grid = std::max<int64_t>(1, std::min(pl.items, (int64_t)st->sm_count * occ));
  PlaneRunParams p{x, y, outer, N, pl.k, pl.items, pl.magic, flags, sc.header, pl.multi ? 1 : 0, (int)inner};
  if (pl.cg) return launched(scan ? launch_planes_cg(p, grid, s) : launch_planes_cg_reduce(op, p, grid, s));
  return launched(scan ? launch_planes_scan((int)inner, p, grid, s)
                       : launch_planes_reduce((int)inner, op, p, grid, s));
}

// Scans of few long planes of 2-8 columns by the look-back form of the
// segmented class runs: one block per tile, the tiles of a plane in scan
// order, each plane's carries from its own look-back tree.  kColLbNoFit when
// its tiles exceed the node words.
int run_planes_lookback(const Provider& pv, const float* x, int64_t outer, int64_t N, int64_t inner, float* y,
                        int flags, cudaStream_t s) {
  DeviceState* st = pv.st;
  const int64_t align = planes_align((int)inner);
  const int64_t tiles = ceil_div(N * inner + align - 1, planes_tile_len((int)inner));  // the most any plane covers
  int64_t total = 0;
  if (mul_overflows(outer, tiles, &total) || total > kMaxLookbackTiles / inner ||
      tiles > (int64_t(1) << (5 * kPlanesLbLevels)))
    return kColLbNoFit;
  Need need;
  need.header = true;
  need.nodes = 2 * total * inner;
  Scratch sc;
  const int rc = acquire(pv, need, &sc, s);
  if (rc) return rc;
  auto* ticket_word = reinterpret_cast<unsigned long long*>(sc.header + 2);
  const int64_t spin = g_opt_spin_limit.load();
  const int64_t lag_opt = g_opt_lookback_lag.load();
  // The lag: 5/4 of this kernel's resident blocks in either direction (a
  // block publishes its tile before it waits on any node).  With 912
  // resident, lags of 960 and 1536 tickets were slower than 1152 on [1, 4e7,
  // 4], [1, 1e8, 2], [1, 5e7, 3] and [64, 1e6, 2], both directions.
  const int64_t resident = (int64_t)st->sm_count * st->occ_planes_lb[inner - 2];
  const int64_t lag_auto = std::max<int64_t>(64, ceil_div(resident * 5 / 4, 64) * 64);
  const int64_t lag = std::min<int64_t>(total, lag_opt > 0 ? lag_opt : lag_auto);
  PlaneLbParams p{x, y, outer, N, tiles, sc.nodes, ticket_word, sc.header,
                  spin > 0 ? spin : kDefaultSpinLimit, g_opt_stall_tile.load(), lag, flags};
  return launched(launch_planes_lookback((int)inner, p, total + lag, s));  // one block per ticket
}

// Scans of few long planes as column groups (k_planes_cg_lb): one block per
// tile of TR whole rows, each column's carry from the plane's look-back
// tree (P node words per tile).  kColLbNoFit when the tiles exceed the node
// words.  The lag as for the plane look-back: 5/4 of the resident blocks.
int run_planes_cg_lookback(const Provider& pv, const float* x, int64_t outer, int64_t N, int64_t inner, float* y,
                           int flags, cudaStream_t s) {
  DeviceState* st = pv.st;
  const int64_t tiles = ceil_div(N, (int64_t)planes_cg_tile_rows((int)inner));
  int64_t total = 0;
  if (mul_overflows(outer, tiles, &total) || total > kMaxLookbackTiles / inner ||
      tiles > (int64_t(1) << (5 * kPlanesLbLevels)))
    return kColLbNoFit;
  Need need;
  need.header = true;
  need.nodes = 2 * total * inner;
  Scratch sc;
  const int rc = acquire(pv, need, &sc, s);
  if (rc) return rc;
  auto* ticket_word = reinterpret_cast<unsigned long long*>(sc.header + 2);
  const int64_t spin = g_opt_spin_limit.load();
  const int64_t lag_opt = g_opt_lookback_lag.load();
  const int64_t resident = (int64_t)st->sm_count * st->occ_planes_cg_lb[cg_instance((int)inner)];
  const int64_t lag_auto = std::max<int64_t>(64, ceil_div(resident * 5 / 4, 64) * 64);
  const int64_t lag = std::min<int64_t>(total, lag_opt > 0 ? lag_opt : lag_auto);
  PlaneLbParams p{x, y, outer, N, tiles, sc.nodes, ticket_word, sc.header,
                  spin > 0 ? spin : kDefaultSpinLimit, g_opt_stall_tile.load(), lag, flags, (int)inner};
  return launched(launch_planes_cg_lookback(p, total + lag, s));
}

int run_cols(const Provider& pv, const float* x, int64_t outer, int64_t reduce, int64_t inner,
             float* out, int op, int epi, cudaStream_t s) {
  DeviceState* st = pv.st;
  const bool vec4 = (inner % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15u) == 0);
  {
    // Narrow rows take the narrow kernel unless a wide shape is forced (sums).
    int vec = 1;
    int64_t fv = g_opt_cols_variant.load();
    const bool wide_forced = op == kOpSum && fv >= 0 && fv < kNumColsVariants;
    PlaneRunPlan pl;
    if ((fv < 0 || fv == kColsPlaneRuns) && g_opt_axis_split.load() <= 0 &&
        (reinterpret_cast<uintptr_t>(x) & 15u) == 0 && plane_run_plan(outer, reduce, inner, &pl, false) &&
        (fv == kColsPlaneRuns || plane_runs_fill(st, pl, outer, reduce, inner, false)))
      return run_planes(pv, pl, x, outer, reduce, inner, out, epi, false, op, s);
    if (fv == kColsPlaneRuns) fv = -1;  // forced on a shape it does not take: the automatic choice
    if ((fv < 0 || fv == kColsShortPlanes) && g_opt_axis_split.load() <= 0) {
      // Narrow planes of at most kShortRowMax rows, many to a chunk.
      const int rc = try_reduce_short_planes(pv, x, outer, reduce, inner, out, op, epi, fv == kColsShortPlanes, s);
      if (rc != kNoPlanes) return rc;
    }
    if (narrow_rows(x, x, inner, &vec) && !wide_forced) {
      // Many small planes: a warp per plane; otherwise a block per (plane, slice).
      const bool warp_form = inner <= 32 * vec && (fv == kColsNarrowWarp ||
                                                   (fv != kColsNarrow && narrow_warp_reduce(st, outer, reduce, inner, vec)));
      if (warp_form) {
        Need need;
        Scratch sc;
        int rc = acquire(pv, need, &sc, s);
        if (rc) return rc;
        const int64_t grid = ceil_div(outer, kThreads / 32);
        if (grid > INT32_MAX) return LIBREDUCE_ERR_OVERFLOW;
        NarrowParams p{x, outer, reduce, inner, 1, reduce, out, nullptr, inner, nullptr, epi, 0};
        return launched(launch_reduce_narrow_warp(vec, op, p, grid, s));
      }
      return run_narrow(pv, x, outer, reduce, inner, out, op, epi, vec, g_opt_axis_split.load(), s);
    }
  }
  int variant = vec4 ? kColsV4W4 : kColsV1W4;
  const int64_t forced_v = g_opt_cols_variant.load();
  if (op == kOpSum && forced_v >= 0 && forced_v < kNumColsVariants) {
    const bool fv4 = forced_v >= kColsV4W1;
    if (!fv4 || vec4) variant = (int)forced_v;
  }
  const int64_t cw = cols_block_width(variant);
  const int64_t col_tiles = ceil_div(inner, cw);
  const int64_t slots = (int64_t)st->sm_count * st->occ_cols[variant][op];
  int64_t base_blocks = 0;
  if (mul_overflows(outer, col_tiles, &base_blocks)) return LIBREDUCE_ERR_OVERFLOW;
  int64_t splits = 1;
  const int64_t forced = g_opt_axis_split.load();
  if (forced > 0) {
    splits = std::min(forced, reduce);
  } else if (base_blocks < slots) {
    // Too few column tiles to fill the GPU: slice the reduce axis so the grid
    // is one wave, as full as possible without spilling into a second one
    // (measured best for a short kernel: no tail, no ramp).
    splits = std::max<int64_t>(1, slots / base_blocks);
    splits = std::min(splits, std::max<int64_t>(1, reduce / 64));  // at least ~64 rows per slice
  }
  int64_t rows_per_split = ceil_div(reduce, splits);
  splits = ceil_div(reduce, rows_per_split);
  if (splits > 1 && (base_blocks > kMaxTickets || splits * base_blocks * cw > kMaxPartials)) {
    // Shrink the split to fit the workspace.
    const int64_t cap = kMaxPartials / (base_blocks * cw);
    if (base_blocks > kMaxTickets || cap < 2) {
      splits = 1;
    } else {
      splits = cap;
    }
    rows_per_split = ceil_div(reduce, splits);
    splits = ceil_div(reduce, rows_per_split);
  }
  int64_t grid = 0;
  if (mul_overflows(base_blocks, splits, &grid) || grid > INT32_MAX) return LIBREDUCE_ERR_OVERFLOW;
  Need need;
  if (splits > 1) {
    need.tickets = base_blocks;
    need.partials = splits * base_blocks * cw;
  }
  Scratch sc;
  int rc = acquire(pv, need, &sc, s);
  if (rc) return rc;
  ColsParams p{x, outer, reduce, inner, (int32_t)col_tiles, (int32_t)splits, rows_per_split,
               out, sc.partials, sc.tickets, epi, 0};
  return launched(launch_reduce_cols(variant, op, p, grid, s));
}

// Public operator -> (kernel operator, epilogue, value of an empty reduction).
struct OpPlan {
  int op;
  int epi;
  float empty;
};
bool plan_op(int public_op, OpPlan* plan) {
  const float inf = __builtin_inff(), nan = __builtin_nanf("");
  switch (public_op) {
    case LIBREDUCE_OP_SUM: *plan = {kOpSum, kEpiNone, 0.f}; return true;
    case LIBREDUCE_OP_MEAN: *plan = {kOpSum, kEpiMean, nan}; return true;
    case LIBREDUCE_OP_MAX: *plan = {kOpMax, kEpiNone, -inf}; return true;
    case LIBREDUCE_OP_MIN: *plan = {kOpMin, kEpiNone, inf}; return true;
    case LIBREDUCE_OP_NORM: *plan = {kOpSumSq, kEpiSqrt, 0.f}; return true;
    default: return false;
  }
}

// Turn an internal status into the public one (a size query is a success).
int finish_status(int rc) { return rc == kQueried ? LIBREDUCE_OK : rc; }

// The reduction behind every reduce entry point: `out[o*inner + i]` is the
// reduction of x[o, :, i] over the middle axis of [outer, reduce, inner].
int reduce_impl(const float* x, int64_t outer, int64_t reduce, int64_t inner, float* out,
                int public_op, Provider pv, cudaStream_t s) {
  OpPlan plan;
  if (!plan_op(public_op, &plan)) return LIBREDUCE_ERR_INVALID_ARG;
  if (outer < 0 || reduce < 0 || inner < 0) return LIBREDUCE_ERR_INVALID_ARG;
  int64_t n_out = 0, total = 0;
  if (mul_overflows(outer, inner, &n_out) || mul_overflows(n_out, reduce, &total) ||
      total > INT64_MAX / 4)
    return LIBREDUCE_ERR_OVERFLOW;
  if (n_out == 0) {
    if (pv.query) *pv.query = 0;
    return LIBREDUCE_OK;
  }
  if (out == nullptr || (x == nullptr && total > 0)) return LIBREDUCE_ERR_INVALID_ARG;
  if (overlaps(x, (size_t)total * sizeof(float), out, (size_t)n_out * sizeof(float)))
    return LIBREDUCE_ERR_ALIAS;
  dbg_call_buffers(x, (size_t)total * sizeof(float), out, (size_t)n_out * sizeof(float));
  int dev = 0;
  int rc = device_state(&pv.st, &dev);
  if (rc) return rc;
  if ((rc = check_buffer(out, (size_t)n_out * sizeof(float), dev))) return rc;
  if (total == 0) {
    Scratch sc;
    if ((rc = acquire(pv, Need{}, &sc, s))) return finish_status(rc);
    if (plan.empty == 0.f) {
      const cudaError_t e = cudaMemsetAsync(out, 0, (size_t)n_out * sizeof(float), s);
      return e == cudaSuccess ? LIBREDUCE_OK : fail_cuda(e);
    }
    return launched(launch_fill(out, n_out, plan.empty, s));
  }
  if ((rc = check_buffer(x, (size_t)total * sizeof(float), dev))) return rc;
  if (inner == 1) {
    if (outer == 1) return finish_status(run_contig(pv, x, 1, reduce, out, plan.op, plan.epi, s));
    if (reduce <= kRowsWarpMaxLen && g_opt_axis_split.load() <= 0) {
      const int64_t form = g_opt_rows_form.load();
      if (form == 2 || (form == 0 && reduce <= kShortReduceMax))
        return finish_status(run_rows_short(pv, x, outer, reduce, out, plan.op, plan.epi, s));
      return finish_status(run_rows_warp(pv, x, outer, reduce, out, plan.op, plan.epi, s));
    }
    return finish_status(run_contig(pv, x, outer, reduce, out, plan.op, plan.epi, s));
  }
  return finish_status(run_cols(pv, x, outer, reduce, inner, out, plan.op, plan.epi, s));
}

// L2-lag form: tickets between a tile's two touches.  In the reverse scan's
// order (write, then publish) the lag must exceed the blocks resident at
// once, or the write of tile t - lag waits on tiles still in flight; past
// ~2000 tiles (64 MiB) the reread misses L2.  Measured on one row of 1e9 with
// 608 resident blocks (4 per SM): reverse 55% at lag 384, 63% at 512, 87% at
// 768, 94-96% at 1024, 87% at 1280, 76% at 1536: 5/3 of the resident blocks.
// The forward scan publishes first and reaches 92% at 640-768 (89% at 1024):
// 5/4 of the resident blocks.  Both in steps of 64.
int64_t lookback_lag(const DeviceState* st, bool mirror, int period = 1) {
  const int64_t resident = (int64_t)st->sm_count * st->occ_lookback_period[period_slot(period)];
  const int64_t lag = mirror ? resident * 5 / 4 : resident * 5 / 3;
  return std::max<int64_t>(64, ceil_div(lag, 64) * 64);
}

// Row scans with float4 tiles read any row as a 16-byte aligned "virtual
// row" (the scan kernels' RowView): they need x and y to share their 16-byte
// misalignment.  The longest virtual row is the row padded by its
// misalignment (the same for every row when N % 4 == 0, else up to 3) and
// rounded up to a multiple of 4.
bool rows_vec4(const float* x, const float* y) {
  return ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
}
// Float4 rows that are not whole aligned float4s run the kernel forms that
// mask the row edges.
bool has_row_edges(const float* x, int64_t N) {
  return N % 4 != 0 || (reinterpret_cast<uintptr_t>(x) & 15u) != 0;
}
int64_t virtual_row_len(const float* x, int64_t N, bool vec4) {
  if (!vec4) return N;
  const int64_t m0 = (int64_t)((reinterpret_cast<uintptr_t>(x) >> 2) & 3);
  return round_up(N + (N % 4 == 0 ? m0 : 3), 4);
}

int run_rscan_lookback(const Provider& pv, const float* x, int64_t rows, int64_t N, float* y,
                       cudaStream_t s, int variant, int flags, int period = 1) {
  const int64_t tile = period == 1 ? lookback_tile(variant) : lookback_tile_period(period);
  const int64_t tiles = ceil_div(virtual_row_len(x, N, variant != kLookbackV1), tile);
  int64_t total = 0;
  if (mul_overflows(rows, tiles, &total) || total > kMaxLookbackTiles / period) return LIBREDUCE_ERR_OVERFLOW;
  Need need;
  need.header = true;
  need.nodes = 2 * total * period;
  Scratch sc;
  int rc = acquire(pv, need, &sc, s);
  if (rc) return rc;
  // Header words 2-3: {ticket counter, epoch} as one 64-bit word; the block
  // with the last ticket resets the counter and advances the epoch.
  auto* ticket_word = reinterpret_cast<unsigned long long*>(sc.header + 2);
  const int64_t spin = g_opt_spin_limit.load();
  const int64_t lag_opt = g_opt_lookback_lag.load();
  const int64_t lag = variant == kLookbackL2
                          ? std::min<int64_t>(total, lag_opt > 0 ? lag_opt
                                                                 : lookback_lag(pv.st, (flags & kScanMirror) != 0, period))
                          : 0;
  if (variant == kLookbackL2 && has_row_edges(x, N)) flags |= kScanRowEdges;
  RScanLookbackParams p{x, y, rows, N, tiles, sc.nodes, ticket_word, sc.header,
                        spin > 0 ? spin : kDefaultSpinLimit, g_opt_stall_tile.load(), lag, flags, period};
  const int64_t grid = total + lag;  // one block per ticket
  return launched(launch_rscan_lookback(variant, p, grid, s));
}

// Reduce-then-scan along rows: tile sums, a reverse exclusive scan of the
// sums (one block per row), then every tile scanned again with its carry.
int run_reduce_then_scan(const Provider& pv, const float* x, int64_t rows, int64_t N, float* y,
                         cudaStream_t s, int flags, bool vec4) {
  const int variant = vec4 ? kTileV4 : kTileV1;
  const int64_t tiles = ceil_div(virtual_row_len(x, N, vec4), tile_scan_len(variant));
  int64_t total = 0;
  if (mul_overflows(rows, tiles, &total) || 2 * total > kMaxPartials || total > INT32_MAX)
    return LIBREDUCE_ERR_OVERFLOW;
  Need need;
  need.partials = 2 * total;
  Scratch sc;
  int rc = acquire(pv, need, &sc, s);
  if (rc) return rc;
  float* sums = sc.partials;
  float* carries = sc.partials + total;
  if (vec4 && has_row_edges(x, N)) flags |= kScanRowEdges;
  TileSumsParams p1{x, rows, N, tiles, sums, flags};
  if ((rc = launched(launch_tile_sums(variant, p1, total, s)))) return rc;
  RScanRowsParams p2{sums, carries, rows, tiles, kScanExclusive};
  if ((rc = launched(launch_rscan_rows(kRScanV1S4, p2, std::min<int64_t>(rows, INT32_MAX), s))))
    return rc;
  TileCarryParams p3{x, y, rows, N, tiles, carries, flags};
  return launched(launch_tile_carry_scan(variant, p3, total, s));
}

// Scans and reductions of many short rows (N <= kShortRowMax): chunks of whole
// rows staged in shared memory, each row handled by a group of G lanes.
struct ShortPlan {
  int lanes, run, stride, rows_per_chunk;
  unsigned long long magic;
};
// Rows of at most `solo` elements: one lane per row, chunks of about
// `target` floats with at least 8 rows where they fit.  Longer rows: groups of
// G lanes (a power of two, 4 to 32) with lane runs of L = ceil(N/G) | 1, and
// chunks that the prefetch covers (at most kShortChunk floats; a longer chunk
// loads its remainder at staging) and that the block's 128/G groups cover in
// one pass at least 3/4 full:
//   rows = kShortChunk / N, at least 4 (one pass of 32-lane groups) and at
//          most 32 (one pass of 4-lane groups), within the shared memory;
//   G    = the largest with rows <= 128/G; if that pass would be less than
//          3/4 full, G doubles and rows = 128/G.
// Measured on scans of 2e8 floats (fraction of copy bandwidth, [rows, N]):
// runs of 25-33 elements in one pass beat runs of 7-17 over two partly idle
// passes ([., 100] 0.96 at G = 4 against 0.69 at G = 16; [., 256] 0.96
// against 0.91), a full pass beats a 3/5 one ([., 160] 0.97 at G = 8 with 16
// rows against 0.88 at G = 4 with 19), chunks of up to 3072 floats beat
// larger ones with a remainder ([., 128] 0.96 against 0.93), and one lane per
// row stays best up to 64 elements (0.97-0.98).
// Where a chunk holds at least the rows that span a whole number of 128-byte
// lines, it is rounded down to a multiple of them, so every chunk starts on a
// line boundary and no line is shared by two blocks.
ShortPlan short_plan(int64_t N, int64_t target, int64_t solo) {
  ShortPlan q{1, (int)N, (int)(N | 1), 1, 0};
  int64_t a = N, b = 32;  // rows per whole number of lines: 32 / gcd(N, 32)
  while (b) {
    const int64_t r = a % b;
    a = b;
    b = r;
  }
  const int64_t line_rows = 32 / a;
  const auto line_round = [&](int64_t rows) { return rows >= line_rows ? rows - rows % line_rows : rows; };
  if (N <= solo) {
    q.rows_per_chunk = (int)line_round(
        std::max<int64_t>(1, std::min<int64_t>(kShortSmem / q.stride, std::max<int64_t>(8, target / N))));
  } else {
    const int64_t fit = kShortSmem / (N + 31);  // rows that fit at the widest stride a group needs
    int64_t rows = std::min<int64_t>(fit, std::min<int64_t>(32, std::max<int64_t>(4, kShortChunk / N)));
    rows = line_round(std::max<int64_t>(1, rows));
    q.lanes = 4;
    while (q.lanes < 32 && 2 * q.lanes * rows <= kShortThreads) q.lanes <<= 1;
    if (q.lanes < 32 && 4 * rows * q.lanes < 3 * kShortThreads) {
      q.lanes <<= 1;
      rows = line_round(kShortThreads / q.lanes);
    }
    q.run = (int)ceil_div(N, q.lanes) | 1;  // odd: the lanes of a row on distinct banks
    // The rows of a warp on distinct banks too: stride = run * lanes (mod 32).
    q.stride = (int)N;
    if (q.lanes < 32)
      while (q.stride % 32 != (q.run * q.lanes) % 32) ++q.stride;
    // 32-lane groups keep stride N: up to a full pass of them where it fits.
    if (q.lanes == 32) rows = std::max<int64_t>(rows, line_round(std::min<int64_t>(4, kShortSmem / q.stride)));
    q.rows_per_chunk = (int)rows;
  }
  q.magic = ((1ull << 32) + (unsigned long long)N - 1) / (unsigned long long)N;
  return q;
}
int64_t short_grid(const DeviceState* st, int64_t rows, const ShortPlan& q) {
  return std::max<int64_t>(1, std::min<int64_t>(ceil_div(rows, q.rows_per_chunk),
                                                4 * (int64_t)st->sm_count * st->occ_rscan_short));
}

// The load form and plan of a short-row launch: 16-byte loads need whole
// float4 rows (N % 4 == 0) and 16-byte aligned pointers; other rows take
// 4-byte loads.  (Copying 16-byte aligned chunks of such rows as float4s was
// measured and was slower: [., 33] 0.69 against 0.96 for scans, 0.49 against
// 0.75 for sums.)  Odd rows up to solo_odd take one lane each: their chunks
// then lie unpadded in shared memory (stride N), so staging needs no row
// index, where lane groups pad every row (scans of [., 99] 0.78 against 0.66;
// from 500 one lane per row is slower).
struct ShortForm {
  ShortPlan q;
  int vec;
};
ShortForm short_form(int64_t N, int64_t solo, int64_t solo_odd, bool aligned16) {
  return {short_plan(N, kShortChunk, N % 2 ? solo_odd : solo), aligned16 && N % 4 == 0 ? kShortLd4 : kShortLd1};
}

int run_rscan_short(const Provider& pv, const float* x, int64_t rows, int64_t N, float* y, cudaStream_t s,
                    int flags) {
  const ShortForm f = short_form(N, kShortScanSolo, kShortScanSoloOdd,
                                 ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0);
  const ShortPlan& q = f.q;
  Scratch sc;
  int rc = acquire(pv, Need{}, &sc, s);
  if (rc) return rc;
  ShortRowsParams p{x, y, rows, (int)N, q.rows_per_chunk, q.stride, q.run, q.magic, flags, 1, 0};
  return launched(launch_rscan_short(q.lanes, f.vec, p, short_grid(pv.st, rows, q), s));
}

// Narrow planes ([outer, N, inner] along N, N <= kShortRowMax): the short-row
// kernels over chunks of whole planes, each staged transposed so that every
// column is a row of N (see lr_rows_short.cu).  The plan is the rows' plan
// for rows of N, its chunk counted in planes (inner rows each) and kept inside
// the shared memory.  ok == false: not even one plane fits.  (A form that
// staged planes in their own layout, a column read `inner` floats apart,
// raised an illegal-address fault on its first 16-byte-load case; the cause
// was not found, and that form is not used.)
struct PlaneForm {
  ShortForm f;
  bool ok;
};
PlaneForm plane_form(int64_t N, int64_t inner, int64_t solo, int64_t solo_odd, bool aligned16) {
  PlaneForm r{short_form(N, solo, solo_odd, false), false};
  ShortPlan& q = r.f.q;
  if (N > kShortRowMax || inner < 2 || inner > kShortPlaneInnerMax) return r;
  int64_t planes = std::max<int64_t>(1, std::min<int64_t>(q.rows_per_chunk / inner, kShortChunk / (N * inner)));
  while (planes > 1 && planes * inner * q.stride > kShortSmem) --planes;
  if (planes * inner * q.stride > kShortSmem) return r;
  // Chunks of whole 128-byte lines where the planes allow (see short_plan).
  int64_t a = N * inner, b = 32;
  while (b) {
    const int64_t t = a % b;
    a = b;
    b = t;
  }
  const int64_t line_planes = 32 / a;
  if (planes >= line_planes) planes -= planes % line_planes;
  q.rows_per_chunk = (int)planes;
  r.f.vec = aligned16 && (N * inner) % 4 == 0 ? kShortLd4 : kShortLd1;
  r.ok = true;
  return r;
}
int64_t plane_grid(const DeviceState* st, int64_t planes, const ShortPlan& q) {
  return std::max<int64_t>(1, std::min<int64_t>(ceil_div(planes, q.rows_per_chunk),
                                                4 * (int64_t)st->sm_count * st->occ_rscan_short));
}
unsigned long long magic_of(int64_t d) { return ((1ull << 32) + (unsigned long long)d - 1) / (unsigned long long)d; }

int run_scan_short_planes(const Provider& pv, const PlaneForm& pf, const float* x, int64_t outer, int64_t N,
                          int64_t inner, float* y, cudaStream_t s, int flags) {
  const ShortPlan& q = pf.f.q;
  Scratch sc;
  int rc = acquire(pv, Need{}, &sc, s);
  if (rc) return rc;
  ShortRowsParams p{x, y, outer, (int)N, q.rows_per_chunk, q.stride, q.run, q.magic, flags, (int)inner,
                    magic_of(inner)};
  return launched(launch_rscan_short(q.lanes, pf.f.vec, p, plane_grid(pv.st, outer, q), s));
}

int run_reduce_short_planes(const Provider& pv, const PlaneForm& pf, const float* x, int64_t outer, int64_t N,
                            int64_t inner, float* out, int op, int epi, cudaStream_t s);

// The automatic choice: planes of at most kShortReducePlaneMax floats; above
// that a warp per plane (or the narrow block kernel) is ahead.  Measured
// (fraction of copy bandwidth, planes against a warp per plane): [400000,
// 100, 3] 0.59 / 0.55, [1e6, 16, 8] 0.67 / 0.21, [100000, 33, 16] 0.57 /
// 0.47; [50000, 512, 2] 0.58 / 0.84, [20000, 1024, 3] 0.60 / 0.73.  `forced`
// takes any plane that fits the shared memory.
constexpr int64_t kShortReducePlaneMax = 768;
int try_reduce_short_planes(const Provider& pv, const float* x, int64_t outer, int64_t N, int64_t inner,
                            float* out, int op, int epi, bool forced, cudaStream_t s) {
  if (N > kShortRowMax || inner < 2 || inner > kShortPlaneInnerMax || (!forced && N * inner > kShortReducePlaneMax))
    return kNoPlanes;
  const PlaneForm pf = plane_form(N, inner, kShortReduceSolo, kShortReduceSoloOdd,
                                  (reinterpret_cast<uintptr_t>(x) & 15u) == 0);
  if (!pf.ok) return kNoPlanes;
  return run_reduce_short_planes(pv, pf, x, outer, N, inner, out, op, epi, s);
}

int run_reduce_short_planes(const Provider& pv, const PlaneForm& pf, const float* x, int64_t outer, int64_t N,
                            int64_t inner, float* out, int op, int epi, cudaStream_t s) {
  const ShortPlan& q = pf.f.q;
  Scratch sc;
  int rc = acquire(pv, Need{}, &sc, s);
  if (rc) return rc;
  ShortRowsParams p{x, out, outer, (int)N, q.rows_per_chunk, q.stride, q.run, q.magic, epi, (int)inner,
                    magic_of(inner)};
  return launched(launch_reduce_short(op, q.lanes, pf.f.vec, p, plane_grid(pv.st, outer, q), s));
}

// Reductions of many short rows (inner == 1, reduce <= kShortRowMax) with the
// same chunks: one float per row.
int run_rows_short(const Provider& pv, const float* x, int64_t rows, int64_t N, float* out, int op, int epi,
                   cudaStream_t s) {
  const ShortForm f = short_form(N, kShortReduceSolo, kShortReduceSoloOdd, (reinterpret_cast<uintptr_t>(x) & 15u) == 0);
  const ShortPlan& q = f.q;
  Scratch sc;
  int rc = acquire(pv, Need{}, &sc, s);
  if (rc) return rc;
  ShortRowsParams p{x, out, rows, (int)N, q.rows_per_chunk, q.stride, q.run, q.magic, epi, 1, 0};
  return launched(launch_reduce_short(op, q.lanes, f.vec, p, short_grid(pv.st, rows, q), s));
}

// Scans along rows (inner == 1).  `flags`: kScanMirror for a forward scan,
// kScanExclusive to leave out each element's own term.  period 2 or 4: each
// row is a narrow plane of that many columns read flat (N = its floats; the
// caller checks that x and y share their 16-byte offset): float4 tiles one
// block per plane, or the L2 look-back for few planes.
int run_rscan_rows(const Provider& pv, const float* x, int64_t rows, int64_t N, float* y,
                   cudaStream_t s, int flags, int period = 1) {
  DeviceState* st = pv.st;
  const bool vec4 = rows_vec4(x, y);
  int variant = vec4 ? kRScanV4S4 : kRScanV1S4;
  const int64_t forced_v = g_opt_rscan_variant.load();
  if (period == 1 && forced_v >= 0 && forced_v < kNumRScanVariants && (forced_v == kRScanV1S4 || vec4))
    variant = (int)forced_v;
  // Few rows cannot fill the GPU one block per row: use the look-back scan,
  // which spreads every row's tiles over all SMs.
  int64_t strategy = g_opt_scan_strategy.load();
  if (strategy == 5 && N > kShortRowMax) strategy = 0;  // rows too long for the short-row form
  if (period != 1 && strategy != 1 && strategy != 2) strategy = 0;  // only these forms take a period
  const int lb_variant = !vec4 ? kLookbackV1 : (strategy == 3 ? kLookbackV4 : kLookbackL2);
  const int64_t lb_tiles = ceil_div(virtual_row_len(x, N, vec4),
                                    period == 1 ? lookback_tile(lb_variant) : lookback_tile_period(period));
  const int64_t row_slots =
      (int64_t)st->sm_count * (period == 1 ? st->occ_rscan[variant] : st->occ_rscan_period[period_slot(period)]);
  const bool lookback_fits = rows <= kMaxLookbackTiles / period / std::max<int64_t>(1, lb_tiles);
  if (strategy == 4) return run_reduce_then_scan(pv, x, rows, N, y, s, flags, vec4);
  if (period == 1 && (strategy == 5 || (strategy == 0 && N <= kShortRowMax)))
    return run_rscan_short(pv, x, rows, N, y, s, flags);
  if ((strategy >= 2 || (strategy == 0 && 4 * rows < row_slots && lb_tiles >= 4)) && lookback_fits)
    return run_rscan_lookback(pv, x, rows, N, y, s, lb_variant, flags, period);
  if (strategy >= 2 && period == 1) return run_rscan_lookback(pv, x, rows, N, y, s, lb_variant, flags);
  Scratch sc;
  int rc = acquire(pv, Need{}, &sc, s);
  if (rc) return rc;
  const int64_t grid = std::min<int64_t>(rows, INT32_MAX);
  if (variant != kRScanV1S4 && has_row_edges(x, N)) flags |= kScanRowEdges;
  RScanRowsParams p{x, y, rows, N, flags, period};
  return launched(launch_rscan_rows(variant, p, grid, s));
}

int run_scan_narrow(const Provider& pv, const float* x, int64_t outer, int64_t N, int64_t inner,
                    float* y, bool reverse, bool exclusive, int vec, bool warp_form, cudaStream_t s);

// Predicted fraction of the copy bandwidth that a column scan reaches with
// `units` equally long blocks, `slots` of them resident at once, a fraction
// lane_eff of the lanes of a column tile holding columns, and `base` the
// fraction the variant reaches on a large, well-shaped case.  Whole waves run
// at full rate; a wave with fewer active warps than kSatFraction of the slots
// (idle lanes counted out) no longer has enough loads in flight to cover the
// memory latency and takes as long as one that has.  A fit to GB300 sweeps of
// [outer, N, inner] from [1, 5000, 4096] to [4096, 256, 64].
double predict_scan_cols(int64_t units, int64_t slots, double lane_eff, double base) {
  constexpr double kSatFraction = 0.6;
  const double floor_a = kSatFraction / lane_eff;
  const int64_t full = units / slots;
  const double rest = (double)(units - full * slots) / (double)slots;
  const double time = (double)full * std::max(1.0, floor_a) + (rest > 0 ? std::max(rest, floor_a) : 0.0);
  return base * ((double)units / (double)slots) / time;
}

// Scans along a strided axis (inner > 1): one block per (o, column tile),
// walking the whole axis.  When those blocks cannot fill the GPU, the axis is
// cut into segments and scanned in three passes: segment sums (the split
// column reduction, keeping every slice), an exclusive scan of the sums along
// the segments (the same scan kernel, one segment), then every segment
// scanned again from its carry.  The block shape and the segment count are
// chosen by predict_scan_cols, the segmented form paying 1.5x for the extra
// read of x.
// Single-pass column scan with a look-back over 256-row x 32-column tiles
// (k_scan_cols_lookback).  Returns kColLbNoFit, before touching anything,
// when the tiles' node words would not fit the look-back region.  The debug
// build never takes it (kColLbNoFit): its checked form of this kernel, with
// the TMA tensor copies, raised a GPU fault whose cause was not found, so it
// stays off the GPU; the three-pass form serves instead.
int run_scan_cols_lookback(const Provider& pv, const float* x, int64_t outer, int64_t N, int64_t inner,
                           float* y, bool reverse, bool exclusive, cudaStream_t s) {
#ifdef LR_DEBUG
  (void)pv, (void)x, (void)outer, (void)N, (void)inner, (void)y, (void)reverse, (void)exclusive, (void)s;
  return kColLbNoFit;
#endif
  const int64_t col_tiles = ceil_div(inner, kColLbCols);
  const int64_t tiles = ceil_div(N, kColLbRows);
  int64_t units = 0, total = 0;
  if (mul_overflows(outer, col_tiles, &units) || mul_overflows(units, tiles, &total) ||
      total > kLookbackWords / (2 * kColLbCols))
    return kColLbNoFit;
  Need need;
  need.header = true;
  need.nodes = 2 * total * kColLbCols;
  Scratch sc;
  int rc = acquire(pv, need, &sc, s);
  if (rc) return rc;
  auto* ticket_word = reinterpret_cast<unsigned long long*>(sc.header + 2);
  const int64_t spin = g_opt_spin_limit.load();
  const int64_t lag_opt = g_opt_lookback_lag.load();
  const int64_t resident = (int64_t)pv.st->sm_count * pv.st->occ_scan_cols_lb;
  // 5/6 of the resident blocks (512 of 608): best or within 0.5% of best
  // from 320 to 768 on [2, 8192, 4096], [1, 16384, 4096], [4, 4096, 2048],
  // [8, 2048, 4096], [1, 65536, 512], [2, 32768, 1024] and [1, 100000, 1024]
  // (768 was 1-5% slower; 448 and below wait on the look-back).
  const int64_t lag = std::min<int64_t>(total, lag_opt > 0 ? lag_opt : std::max<int64_t>(64, ceil_div(resident * 5 / 6, 64) * 64));
  ScanColsLookbackParams p{x, y, outer, N, inner, col_tiles, tiles, sc.nodes, ticket_word, sc.header,
                           spin > 0 ? spin : kDefaultSpinLimit, g_opt_stall_tile.load(), lag,
                           reverse ? 1 : 0, exclusive ? 1 : 0};
  // float4 items need whole aligned float4s in every row of x and y.
  const bool vec4 = inner % 4 == 0 && ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
  return launched(launch_scan_cols_lookback(vec4 ? 4 : 1, p, total + lag, s));
}

int run_scan_cols(const Provider& pv, const float* x, int64_t outer, int64_t N, int64_t inner,
                  float* y, bool reverse, bool exclusive, cudaStream_t s) {
  DeviceState* st = pv.st;
  {
    int nvec = 1;
    int64_t fv = g_opt_scan_cols_variant.load();
    PlaneRunPlan pl;
    if ((fv < 0 || fv == kScanColsPlaneRuns) && g_opt_axis_split.load() <= 0 &&
        ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
        plane_run_plan(outer, N, inner, &pl, true) && (fv == kScanColsPlaneRuns || plane_runs_fill(st, pl, outer, N, inner, true)))
      return run_planes(pv, pl, x, outer, N, inner, y, (reverse ? 0 : kScanMirror) | (exclusive ? kScanExclusive : 0),
                        true, kOpSum, s);
    if ((fv < 0 || fv == kScanColsPlaneLookback) && g_opt_axis_split.load() <= 0 &&
        ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
        plane_run_plan(outer, N, inner, &pl, true) && pl.cg &&
        (fv == kScanColsPlaneLookback ||
         (pl.items < st->sm_count && N >= 2 * planes_cg_tile_rows((int)inner) && !(inner % 32 == 0 && inner >= 64) &&
          !(inner <= kPlanesMaxP && planes_run_len((int)inner) == 36)))) {
      // Few long planes of 7-128 columns: column-group tiles over blocks,
      // carries by look-back (fraction of copy bandwidth against the
      // automatic choice before: [32, 5e5, 9] 0.53 / 0.23, [100, 1e5, 10]
      // 0.67 / 0.24, [64, 2e5, 13] 0.55 / 0.29, [1, 1e7, 16] 0.73 / 0.60,
      // [4, 2e6, 20] 0.62 / 0.46, [1, 4e6, 31] 0.51 / 0.32, [100, 50000, 32]
      // 0.86 / 0.76).  6 columns keep the plane look-back's runs ([16, 1e6,
      // 6] 0.67 / 0.60), 64 and 128 the column look-back's whole 32-column
      // tiles.
      const int rc = run_planes_cg_lookback(pv, x, outer, N, inner, y,
                                            (reverse ? 0 : kScanMirror) | (exclusive ? kScanExclusive : 0), s);
      if (rc != kColLbNoFit) return rc;
    }
    if ((fv < 0 || fv == kScanColsPlaneLookback) && g_opt_axis_split.load() <= 0 &&
        ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
        plane_run_plan(outer, N, inner, &pl, true, false) && !pl.multi && inner <= kPlanesMaxP &&
        (fv == kScanColsPlaneLookback || plane_runs_split(st, pl, N, inner))) {
      // Few long planes: each plane's tiles over blocks, carries by look-back.
      const int rc = run_planes_lookback(pv, x, outer, N, inner, y,
                                         (reverse ? 0 : kScanMirror) | (exclusive ? kScanExclusive : 0), s);
      if (rc != kColLbNoFit) return rc;
    }
    if (fv == kScanColsPlaneRuns || fv == kScanColsPlaneLookback) fv = -1;  // forced on a shape it does not take
    if ((inner == 2 || inner == 4) && rows_vec4(x, y) && g_opt_axis_split.load() <= 0 &&
        (fv == kScanColsPeriodRows || (fv < 0 && inner == 2 && N * inner >= kPeriodRowsMin))) {
      // Planes of 2 or 4 columns: each plane read flat as a row whose
      // elements fall into `inner` column classes, scanned by the row
      // kernels (float4 tiles one block per plane, or the L2 look-back).
      // The automatic choice for 2 columns (fraction of copy bandwidth
      // against the best other form: [16384, 4096, 2] 0.79 / 0.50, [12000,
      // 2048, 2] 0.73 / 0.49, [1, 1e8, 2] 0.55 / 0.38, [64, 1e6, 2] 0.57 /
      // 0.35).  With 4 columns every float4 holds one row, the per-class
      // lane scans (4 per item) bound it by shuffle throughput, and the
      // other forms are ahead ([1, 4e7, 4] 0.43 / 0.53, [8192, 1024, 4] 0.48
      // / 0.50): forced only.
      return run_rscan_rows(pv, x, outer, N * inner, y, s,
                            (reverse ? 0 : kScanMirror) | (exclusive ? kScanExclusive : 0), (int)inner);
    }
    if ((fv == kScanColsShortPlanes ||
         (fv < 0 && inner <= kShortPlaneAutoInnerMax && (inner <= 32 || inner % 4 == 0))) &&
        g_opt_axis_split.load() <= 0 && N <= kShortRowMax && inner <= kShortPlaneInnerMax) {
      // Narrow planes of at most kShortRowMax rows, whole planes to a chunk:
      // ahead of the narrow kernels wherever a plane fits (fraction of copy
      // bandwidth, planes against the better narrow form: [400000, 100, 3]
      // 0.52 / 0.26, [50000, 512, 2] 0.54 / 0.40, [12000, 2048, 2] 0.49 /
      // 0.46, [30000, 100, 32] 0.53 / 0.45).  Above 64 columns, and above 32
      // when the rows are not whole float4s, the wide column scan is ahead
      // ([640, 1000, 100] 0.69 / 0.57, [500, 1000, 128] 0.85 / 0.71,
      // [15000, 100, 47] 0.69 / 0.44, [20000, 100, 33] 0.53 / 0.46): forced
      // only.
      const PlaneForm pf = plane_form(N, inner, kShortScanSolo, kShortScanSoloOdd,
                                      ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0);
      if (pf.ok)
        return run_scan_short_planes(pv, pf, x, outer, N, inner, y, s,
                                     (reverse ? 0 : kScanMirror) | (exclusive ? kScanExclusive : 0));
    }
    // Scalar narrow rows of more than 32 columns (odd widths) and float4 ones
    // of more than 64 go to the wide column scan unless forced ([3000, 300,
    // 33] 0.62 against 0.25, [2000, 500, 65] 0.63 against 0.25; from 17
    // columns on it was already ahead: [3764, 1000, 17] 0.41 / 0.27; float4
    // rows [2604, 256, 96] 0.96 / 0.66, [500, 1000, 128] 0.85 / 0.71 for the
    // best wide variant).
    if (narrow_rows(x, y, inner, &nvec) && (fv >= 0 || (nvec == 4 ? inner <= 64 : inner <= 32)) &&
        (fv < 0 || fv == kScanColsNarrow || fv == kScanColsNarrowWarp || fv == kScanColsShortPlanes ||
         fv == kScanColsPeriodRows)) {
      // The block form walks tiles of T rows; a plane of fewer than T/2 rows
      // would leave most of its threads idle: a warp per plane instead
      // (measured on [100000, 100, 3]: 25% against 4% of copy bandwidth; on
      // larger planes the block form is ahead, e.g. 66% against 20% on
      // [1000, 10000, 8]).
      const bool warp_form = inner <= 32 * nvec && (fv == kScanColsNarrowWarp ||
                                                    (fv < 0 && 2 * N < scan_narrow_tile_rows(nvec, inner)));
      return run_scan_narrow(pv, x, outer, N, inner, y, reverse, exclusive, nvec, warp_form, s);
    }
  }
  const bool vec4 = (inner % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) &&
                    ((reinterpret_cast<uintptr_t>(y) & 15u) == 0);
  const int64_t forced_v = g_opt_scan_cols_variant.load();
  const int64_t forced = g_opt_axis_split.load();
  // Fractions of the copy bandwidth each shape reaches on [128, 4096, 4096]
  // (the scalar shape: 0.75 on [128, 4096, 4095], whose rows are not 16-byte
  // aligned).
  const double base[kNumScanColsVariants] = {vec4 ? 0.906 : 0.75, 0.976, 0.977};
  const bool force = forced_v >= 0 && forced_v < kNumScanColsVariants && (!scan_cols_vec4((int)forced_v) || vec4);
  int variant = vec4 ? kScanColsV4 : kScanColsV1;
  int64_t segs = 1;
  double best = -1.0;
  for (int v = 0; v < kNumScanColsVariants; ++v) {
    if (force ? v != forced_v : (scan_cols_vec4(v) && !vec4)) continue;
    const int64_t cw = scan_cols_block_width(v);
    int64_t units = 0;
    if (mul_overflows(outer, ceil_div(inner, cw), &units)) return LIBREDUCE_ERR_OVERFLOW;
    const int64_t slots = (int64_t)st->sm_count * st->occ_scan_cols[v];
    const double lane_eff = (double)inner / (double)(ceil_div(inner, cw) * cw);
    int64_t cand[2] = {1, 1};
    if (forced > 0) cand[0] = cand[1] = std::min(forced, N);
    else cand[1] = std::min(ceil_div(4 * slots, units), std::max<int64_t>(1, N / (4 * scan_cols_tile_rows(v))));
    for (int64_t sg : cand) {
      double pred = predict_scan_cols(units * sg, slots, lane_eff, base[v]);
      if (sg > 1) pred /= 1.5;
      if (pred > best) {
        best = pred;
        variant = v;
        segs = sg;
      }
    }
  }
  // Where the blocks of one unit each would not fill the GPU, the single-pass
  // look-back replaces the three-pass segmented form (unless a variant or a
  // split is forced).
  if (forced_v == kScanColsLookback || (segs > 1 && forced_v < 0 && forced <= 0)) {
    const int rc = run_scan_cols_lookback(pv, x, outer, N, inner, y, reverse, exclusive, s);
    if (rc != kColLbNoFit) return rc;
  }
  const int64_t units = outer * ceil_div(inner, scan_cols_block_width(variant));
  // The segment sums come from the split column reduction, whose column tiles
  // are padded to its block width; sums and carries must fit the library's
  // partials: take as many segments as fit, or none.  (The sums pass keeps
  // its slices and takes no tickets.)
  const int cvariant = vec4 ? kColsV4W4 : kColsV1W4;
  const int64_t cw = cols_block_width(cvariant);
  const int64_t col_tiles = ceil_div(inner, cw);
  const int64_t inner_pad = col_tiles * cw;
  if (segs > 1) {
    const int64_t cap = kMaxPartials / (2 * outer * inner_pad);
    segs = cap < 2 ? 1 : std::min(segs, cap);
  }
  int64_t seg_len = ceil_div(N, segs);
  segs = ceil_div(N, seg_len);
  Need need;
  if (segs > 1) need.partials = 2 * outer * segs * inner_pad;
  Scratch sc;
  int rc = acquire(pv, need, &sc, s);
  if (rc) return rc;
  const auto grid_for = [](int64_t blocks) { return std::max<int64_t>(1, std::min<int64_t>(blocks, INT32_MAX)); };
  if (segs == 1) {
    ScanColsParams p{x, y, outer, N, inner, reverse ? 1 : 0, exclusive ? 1 : 0, nullptr, 1, N, 0};
    return launched(launch_scan_cols(variant, p, grid_for(units), s));
  }
  float* sums = sc.partials;                               // [outer, segs, inner_pad]
  float* carries = sc.partials + outer * segs * inner_pad;  // same shape
  ColsParams p1{x, outer, N, inner, (int32_t)col_tiles, (int32_t)segs, seg_len,
                nullptr, sums, nullptr, kEpiNone, 1};
  if ((rc = launched(launch_reduce_cols(cvariant, kOpSum, p1, outer * col_tiles * segs, s)))) return rc;
  ScanColsParams p2{sums, carries, outer, segs, inner_pad, reverse ? 1 : 0, 1, nullptr, 1, segs, 0};
  const int64_t units2 = outer * ceil_div(inner_pad, scan_cols_block_width(kScanColsV4));
  if ((rc = launched(launch_scan_cols(kScanColsV4, p2, grid_for(units2), s)))) return rc;
  ScanColsParams p3{x, y, outer, N, inner, reverse ? 1 : 0, exclusive ? 1 : 0, carries, segs, seg_len,
                    inner_pad};
  return launched(launch_scan_cols(variant, p3, grid_for(units * segs), s));
}

// Scans along a strided axis with narrow rows: one block per (o, segment),
// walking the segment in shared-memory tiles.  When outer alone cannot fill
// the GPU the axis is cut into segments and scanned in three passes, as in
// run_scan_cols: segment sums from the narrow reduction (kept slices, rows
// padded to a multiple of 4 floats with zeros), an exclusive scan of the sums
// along the segments, then every segment rescanned from its carry.
int run_scan_narrow(const Provider& pv, const float* x, int64_t outer, int64_t N, int64_t inner,
                    float* y, bool reverse, bool exclusive, int vec, bool warp_form, cudaStream_t s) {
  DeviceState* st = pv.st;
  int64_t tpr = 1;
  while (tpr * vec < inner) tpr <<= 1;
  // Units are warps (warp form) or blocks; rows one unit walks per step.
  const int64_t per_block = warp_form ? kThreads / 32 : 1;
  const int64_t slots = (int64_t)st->sm_count * per_block *
                        (warp_form ? st->occ_scan_narrow_warp[vec == 4] : st->occ_scan_narrow[vec == 4]);
  const int64_t tile_rows = warp_form ? 8 * (32 / tpr) : scan_narrow_tile_rows(vec, inner);
  const double lane_eff = (double)inner / (double)(tpr * vec);
  const int64_t part_stride = round_up(inner, 4);
  int64_t segs = 1;
  const int64_t forced = g_opt_axis_split.load();
  if (forced > 0) {
    segs = std::min(forced, N);
  } else {
    const int64_t cand = std::min(ceil_div(4 * slots, outer), std::max<int64_t>(1, N / (4 * tile_rows)));
    if (cand > 1 && predict_scan_cols(outer * cand, slots, lane_eff, 1.0) / 1.5 >
                        predict_scan_cols(outer, slots, lane_eff, 1.0))
      segs = cand;
  }
  // Where the planes must be cut into segments and the float4 columns (x, y
  // aligned) fill 32-column tiles (at least 90% of their lanes), the
  // single-pass column look-back
  // beats the three passes (measured: [2, 4e6, 128] 0.70 against 0.62,
  // [2, 2e6, 96] 0.66 against 0.50, [8, 2e6, 32] 0.67 against 0.65; with
  // idle lanes it loses, e.g. [2, 4e6, 36] 0.40 against 0.44).
  if (segs > 1 && forced <= 0 && !warp_form && vec == 4 && g_opt_scan_cols_variant.load() < 0 &&
      10 * inner >= 9 * kColLbCols * ceil_div(inner, kColLbCols)) {
    const int rc = run_scan_cols_lookback(pv, x, outer, N, inner, y, reverse, exclusive, s);
    if (rc != kColLbNoFit) return rc;
  }
  if (segs > 1) {
    const int64_t cap = kMaxPartials / (2 * outer * part_stride);
    segs = cap < 2 ? 1 : std::min(segs, cap);
  }
  const int64_t seg_len = ceil_div(N, segs);
  segs = ceil_div(N, seg_len);
  int64_t units = 0;
  if (mul_overflows(outer, segs, &units)) return LIBREDUCE_ERR_OVERFLOW;
  const auto grid_for = [](int64_t blocks) { return std::max<int64_t>(1, std::min<int64_t>(blocks, INT32_MAX)); };
  Need need;  // also answers a size query when nothing is needed
  if (segs > 1) need.partials = 2 * outer * segs * part_stride;
  Scratch sc;
  int rc = acquire(pv, need, &sc, s);
  if (rc) return rc;
  const auto scan = [&](const ScanColsParams& q, int v) {
    return warp_form ? launch_scan_narrow_warp(v, q, grid_for(ceil_div(q.outer * q.segs, per_block)), s)
                     : launch_scan_narrow(v, q, grid_for(q.outer * q.segs), s);
  };
  if (segs == 1) {
    ScanColsParams p{x, y, outer, N, inner, reverse ? 1 : 0, exclusive ? 1 : 0, nullptr, 1, N, 0};
    return launched(scan(p, vec));
  }
  float* sums = sc.partials;                                 // [outer, segs, part_stride]
  float* carries = sc.partials + outer * segs * part_stride;  // same shape
  NarrowParams p1{x, outer, N, inner, segs, seg_len, nullptr, sums, part_stride, nullptr, kEpiNone, 1};
  if ((rc = launched(launch_reduce_narrow(vec, kOpSum, p1, units, s)))) return rc;
  ScanColsParams p2{sums, carries, outer, segs, part_stride, reverse ? 1 : 0, 1, nullptr, 1, segs, 0};
  if ((rc = launched(scan(p2, 4)))) return rc;
  ScanColsParams p3{x, y, outer, N, inner, reverse ? 1 : 0, exclusive ? 1 : 0, carries, segs, seg_len,
                    part_stride};
  return launched(scan(p3, vec));
}

// The cumulative sum behind every scan entry point.
int cumsum_impl(const float* x, int64_t outer, int64_t N, int64_t inner, float* y, unsigned flags,
                Provider pv, cudaStream_t s) {
  if (outer < 0 || N < 0 || inner < 0) return LIBREDUCE_ERR_INVALID_ARG;
  if (flags & ~(LIBREDUCE_SCAN_REVERSE | LIBREDUCE_SCAN_EXCLUSIVE)) return LIBREDUCE_ERR_INVALID_ARG;
  int64_t rows = 0, total = 0;
  if (mul_overflows(outer, inner, &rows) || mul_overflows(rows, N, &total) || total > INT64_MAX / 4)
    return LIBREDUCE_ERR_OVERFLOW;
  if (total == 0) {
    if (pv.query) *pv.query = 0;
    return LIBREDUCE_OK;
  }
  if (x == nullptr || y == nullptr) return LIBREDUCE_ERR_INVALID_ARG;
  const size_t bytes = (size_t)total * sizeof(float);
  if (overlaps(x, bytes, y, bytes)) return LIBREDUCE_ERR_ALIAS;
  dbg_call_buffers(x, bytes, y, bytes);
  int dev = 0;
  int rc = device_state(&pv.st, &dev);
  if (rc) return rc;
  if ((rc = check_buffer(x, bytes, dev))) return rc;
  if ((rc = check_buffer(y, bytes, dev))) return rc;
  const bool reverse = (flags & LIBREDUCE_SCAN_REVERSE) != 0;
  const bool exclusive = (flags & LIBREDUCE_SCAN_EXCLUSIVE) != 0;
  if (inner == 1)
    return finish_status(run_rscan_rows(
        pv, x, outer, N, y, s, (reverse ? 0 : kScanMirror) | (exclusive ? kScanExclusive : 0)));
  return finish_status(run_scan_cols(pv, x, outer, N, inner, y, reverse, exclusive, s));
}

// Provider for the *_ws entry points: a size query when ws is null, else the
// caller's buffer (device memory of the current device, 256-byte aligned).
int ws_provider(void* ws, size_t* ws_bytes, Provider* pv) {
  if (ws_bytes == nullptr) return LIBREDUCE_ERR_INVALID_ARG;
  if (ws == nullptr) {
    pv->query = ws_bytes;
    return LIBREDUCE_OK;
  }
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return LIBREDUCE_ERR_INVALID_ARG;
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  int rc = check_buffer(ws, *ws_bytes, dev);
  if (rc) return rc;
  pv->ws = static_cast<char*>(ws);
  pv->ws_bytes = *ws_bytes;
  return LIBREDUCE_OK;
}

}  // namespace

int check_device_buffer(const void* p, size_t bytes, int dev) { return check_buffer(p, bytes, dev); }

cudaError_t dbg_register_ranges(cudaStream_t s, const void* const* p, const size_t* bytes, int n) {
#ifdef LR_DEBUG
  LrDebug h{};
  for (int i = 0; i < kDbgRanges && i < n; ++i) {
    if (p[i] == nullptr || bytes[i] == 0) continue;
    h.lo[i] = reinterpret_cast<unsigned long long>(p[i]);
    h.hi[i] = h.lo[i] + bytes[i];
  }
  // The ranges only (the findings stay until libreduce_check reads them).
  return cudaMemcpyToSymbolAsync(g_lr_debug, &h, offsetof(LrDebug, flags), 0, cudaMemcpyHostToDevice, s);
#else
  (void)s;
  (void)p;
  (void)bytes;
  (void)n;
  return cudaSuccess;
#endif
}

// Debug builds: read and clear the findings after a synchronisation; returns
// LIBREDUCE_ERR_BOUNDS when a check failed since the last read.
int dbg_take_findings() {
#ifdef LR_DEBUG
  LrDebug h{};
  cudaError_t e = cudaMemcpyFromSymbol(&h, g_lr_debug, sizeof(h));
  if (e != cudaSuccess) return fail_cuda(e);
  if (h.flags == 0) return LIBREDUCE_OK;
  g_dbg_last_bad = h.first_bad & ~1ull;
  const unsigned zero[4] = {0, 0, 0, 0};
  static_assert(offsetof(LrDebug, first_bad) + sizeof(unsigned long long) - offsetof(LrDebug, flags) <= sizeof(zero),
                "findings fit the cleared words");
  e = cudaMemcpyToSymbol(g_lr_debug, zero, sizeof(LrDebug) - offsetof(LrDebug, flags), offsetof(LrDebug, flags));
  if (e != cudaSuccess) return fail_cuda(e);
  return LIBREDUCE_ERR_BOUNDS;
#else
  return LIBREDUCE_OK;
#endif
}
int record_cuda_error(cudaError_t e) { return fail_cuda(e); }
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

}  // namespace lr

using namespace lr;

extern "C" {

int reduce_sum_f32(const float* x, int64_t n, float* out, libreduce_stream_t stream) {
  return reduce_f32(x, n, out, LIBREDUCE_OP_SUM, stream);
}

int reduce_f32(const float* x, int64_t n, float* out, int op, libreduce_stream_t stream) {
  if (n < 0 || out == nullptr || (x == nullptr && n > 0)) return LIBREDUCE_ERR_INVALID_ARG;
  if (n > INT64_MAX / 4) return LIBREDUCE_ERR_OVERFLOW;
  return reduce_impl(x, 1, n, 1, out, op, Provider{}, reinterpret_cast<cudaStream_t>(stream));
}

int reduce_axis_f32(const float* x, int64_t outer, int64_t reduce, int64_t inner, float* out,
                    libreduce_stream_t stream) {
  return reduce_impl(x, outer, reduce, inner, out, LIBREDUCE_OP_SUM, Provider{},
                     reinterpret_cast<cudaStream_t>(stream));
}

int reduce_axis_op_f32(const float* x, int64_t outer, int64_t reduce, int64_t inner, float* out,
                       int op, libreduce_stream_t stream) {
  return reduce_impl(x, outer, reduce, inner, out, op, Provider{}, reinterpret_cast<cudaStream_t>(stream));
}

int reduce_axis_op_ws_f32(const float* x, int64_t outer, int64_t reduce, int64_t inner, float* out,
                          int op, void* ws, size_t* ws_bytes, libreduce_stream_t stream) {
  Provider pv;
  int rc = ws_provider(ws, ws_bytes, &pv);
  if (rc) return rc;
  return reduce_impl(x, outer, reduce, inner, out, op, pv, reinterpret_cast<cudaStream_t>(stream));
}

int reverse_cumsum_f32(const float* x, int64_t rows, int64_t N, float* y,
                       libreduce_stream_t stream) {
  return cumsum_impl(x, rows, N, 1, y, LIBREDUCE_SCAN_REVERSE, Provider{},
                     reinterpret_cast<cudaStream_t>(stream));
}

int cumsum_f32(const float* x, int64_t outer, int64_t N, int64_t inner, float* y, unsigned flags,
               libreduce_stream_t stream) {
  return cumsum_impl(x, outer, N, inner, y, flags, Provider{}, reinterpret_cast<cudaStream_t>(stream));
}

int cumsum_ws_f32(const float* x, int64_t outer, int64_t N, int64_t inner, float* y, unsigned flags,
                  void* ws, size_t* ws_bytes, libreduce_stream_t stream) {
  Provider pv;
  int rc = ws_provider(ws, ws_bytes, &pv);
  if (rc) return rc;
  return cumsum_impl(x, outer, N, inner, y, flags, pv, reinterpret_cast<cudaStream_t>(stream));
}

int libreduce_check(libreduce_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  DeviceState* st = nullptr;
  int rc = device_state(&st, nullptr);
  if (rc) return rc;
  if ((rc = dbg_take_findings())) return rc;
  if (!st->ws) return LIBREDUCE_OK;
  unsigned word = 0;
  e = cudaMemcpyAsync(&word, st->err_word, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  if (word == 0) return LIBREDUCE_OK;
  // Clear the error and abort words and the look-back ticket counter, which an
  // interrupted launch may have left behind.
  e = cudaMemsetAsync(st->err_word, 0, 3 * sizeof(unsigned), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  return LIBREDUCE_ERR_TIMEOUT;
}

int libreduce_check_ws(void* ws, libreduce_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  if (ws == nullptr) return LIBREDUCE_ERR_INVALID_ARG;
  if (const int rc = dbg_take_findings()) return rc;
  unsigned word = 0;
  e = cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  if (word == 0) return LIBREDUCE_OK;
  e = cudaMemsetAsync(ws, 0, 3 * sizeof(unsigned), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  return LIBREDUCE_ERR_TIMEOUT;
}

const char* libreduce_strerror(int status) {
  switch (status) {
    case LIBREDUCE_OK: return "ok";
    case LIBREDUCE_ERR_INVALID_ARG: return "invalid argument";
    case LIBREDUCE_ERR_OVERFLOW: return "size overflow or beyond the workspace limits";
    case LIBREDUCE_ERR_ALIAS: return "output overlaps input";
    case LIBREDUCE_ERR_CUDA: return "CUDA runtime error";
    case LIBREDUCE_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    case LIBREDUCE_ERR_BOUNDS: return "debug build: a kernel access outside its call's buffers was skipped";
    default: return "unknown status";
  }
}

int libreduce_last_cuda_error(void) { return t_last_cuda_error; }

int64_t libreduce_launch_count(void) { return g_launches.load(); }

int libreduce_debug_build(void) {
#ifdef LR_DEBUG
  return 1;
#else
  return 0;
#endif
}

uint64_t libreduce_debug_bad_address(void) { return g_dbg_last_bad.load(); }

int libreduce_set_option(int option, int64_t value) {
  switch (option) {
    case LIBREDUCE_OPT_SCAN_STRATEGY:
      if (value < 0 || value > 5) return LIBREDUCE_ERR_INVALID_ARG;
      g_opt_scan_strategy = value;
      return LIBREDUCE_OK;
    case LIBREDUCE_OPT_AXIS_SPLIT:
      if (value < 0 || value > INT32_MAX) return LIBREDUCE_ERR_INVALID_ARG;
      g_opt_axis_split = value;
      return LIBREDUCE_OK;
    case LIBREDUCE_OPT_SPIN_LIMIT:
      if (value < 0) return LIBREDUCE_ERR_INVALID_ARG;
      g_opt_spin_limit = value;
      return LIBREDUCE_OK;
    case LIBREDUCE_OPT_STALL_TILE:
      if (value < -1) return LIBREDUCE_ERR_INVALID_ARG;
      g_opt_stall_tile = value;
      return LIBREDUCE_OK;
    case LIBREDUCE_OPT_CONTIG_VARIANT:
      if (value < -1 || value >= kNumContigVariants) return LIBREDUCE_ERR_INVALID_ARG;
      g_opt_contig_variant = value;
      return LIBREDUCE_OK;
    case LIBREDUCE_OPT_COLS_VARIANT:
      if (value < -1 || value > kColsPlaneRuns) return LIBREDUCE_ERR_INVALID_ARG;
      g_opt_cols_variant = value;
      return LIBREDUCE_OK;
    case LIBREDUCE_OPT_RSCAN_VARIANT:
      if (value < -1 || value >= kNumRScanVariants) return LIBREDUCE_ERR_INVALID_ARG;
      g_opt_rscan_variant = value;
      return LIBREDUCE_OK;
    case LIBREDUCE_OPT_SCAN_COLS_VARIANT:
      if (value < -1 || value > kScanColsPlaneLookback) return LIBREDUCE_ERR_INVALID_ARG;
      g_opt_scan_cols_variant = value;
      return LIBREDUCE_OK;
    case LIBREDUCE_OPT_ROWS_FORM:
      if (value < 0 || value > 2) return LIBREDUCE_ERR_INVALID_ARG;
      g_opt_rows_form = value;
      return LIBREDUCE_OK;
    case LIBREDUCE_OPT_LOOKBACK_LAG:
      if (value < 0 || value > (1 << 20)) return LIBREDUCE_ERR_INVALID_ARG;
      g_opt_lookback_lag = value;
      return LIBREDUCE_OK;
    case LIBREDUCE_OPT_WAVES:
      if (value < 0 || value > 64) return LIBREDUCE_ERR_INVALID_ARG;
      g_opt_waves = value;
      return LIBREDUCE_OK;
    default:
      return LIBREDUCE_ERR_INVALID_ARG;
  }
}

}  // extern "C"
