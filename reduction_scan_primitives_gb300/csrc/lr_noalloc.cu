// lr_noalloc.cu -- reduce_sum_f32_noalloc: the 1D sum for callers that cannot
// allocate device memory.
//
// reduce_sum_f32 takes its partial sums and ticket from a workspace the
// library allocates with cudaMalloc on first use.  Some callers cannot let
// that happen: code running where device allocation is forbidden or must be
// accounted for up front (inside a custom allocator, or a service whose
// device memory is capped and budgeted before it starts).  This entry point
// runs the same kernel with its scratch in a fixed static device array, so a
// call allocates nothing.
//
// The array (g_noalloc_scratch) lives in this file.  Host code cannot use its
// name as a device address, so set-up asks the runtime for the address with
// cudaGetSymbolAddress, once per device (and again if that device's context
// was replaced, e.g. after cudaDeviceReset) with that device current, and
// passes it to the kernel.  The first call on a device does this set-up; make
// that first call before any stream capture.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "libreduce.h"
#include "lr_contig.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

constexpr int64_t kNoAllocMaxBlocks = 16384;              // partial sums the array holds
constexpr int64_t kNoAllocMaxChunk = int64_t(1) << 22;    // floats per block, at most
constexpr int64_t kNoAllocMaxN = kNoAllocMaxBlocks * kNoAllocMaxChunk;  // 2^36 floats
constexpr size_t kTicketBytes = 256;
constexpr size_t kScratchBytes = kTicketBytes + sizeof(float) * kNoAllocMaxBlocks;  // 64.25 KiB
constexpr int64_t kMinChunkNA = 8192;
constexpr int64_t kTargetChunkNA = 65536;
constexpr int kMaxDevicesNA = 64;

// Scratch shared by every call on a device: [ticket (4 B) | 252 bytes spare |
// partial sums].  Every GPU that loads the library holds it until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct NoAllocDevice {
  bool ready = false;
  CUcontext ctx = nullptr;           // the context the address belongs to
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
  int64_t slots = 0;                 // resident blocks of the kernel
};

std::mutex g_na_mu;
NoAllocDevice g_na_dev[kMaxDevicesNA];

// The driver's cuCtxGetCurrent through the runtime (no link against the
// driver library); null where unavailable.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static const CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  return fn;
}

// Per-device set-up, with `dev` current: the array's device address and the
// kernel's occupancy.  A context replaced since (the device was reset) loads
// the module again, possibly at another address, so set-up runs again then.
// Allocates nothing.
int setup(int dev, NoAllocDevice** out) {
  std::lock_guard<std::mutex> lk(g_na_mu);
  NoAllocDevice& d = g_na_dev[dev];
  CUcontext ctx = nullptr;
  if (CtxGetCurrentFn get = ctx_get_current()) {
    if (get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  }
  if (!d.ready || ctx != d.ctx) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return record_cuda_error(e);
    int sms = 0, occ = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_reduce_contig<16, OpSum>, kThreads, 0);
    if (e != cudaSuccess) return record_cuda_error(e);
    d.scratch = static_cast<unsigned char*>(p);
    d.slots = (int64_t)sms * std::max(1, occ);
    d.ctx = ctx;
    d.ready = true;
  }
  *out = &d;
  return LIBREDUCE_OK;
}

}  // namespace
}  // namespace lr

using namespace lr;

extern "C" int reduce_sum_f32_noalloc(const float* x, int64_t n, float* out,
                                      libreduce_stream_t stream) {
  if (n < 0 || out == nullptr || (x == nullptr && n > 0)) return LIBREDUCE_ERR_INVALID_ARG;
  if (n > kNoAllocMaxN) return LIBREDUCE_ERR_OVERFLOW;
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), o0 = reinterpret_cast<uintptr_t>(out);
  if (n > 0 && o0 < x0 + (uint64_t)n * sizeof(float) && x0 < o0 + sizeof(float))
    return LIBREDUCE_ERR_ALIAS;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevicesNA) return LIBREDUCE_ERR_INVALID_ARG;
  int rc = check_device_buffer(out, sizeof(float), dev);
  if (rc) return rc;
  if (n > 0 && (rc = check_device_buffer(x, (size_t)n * sizeof(float), dev))) return rc;
  NoAllocDevice* d = nullptr;
  if ((rc = setup(dev, &d))) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (n == 0) {
    e = cudaMemsetAsync(out, 0, sizeof(float), s);
    return e == cudaSuccess ? LIBREDUCE_OK : record_cuda_error(e);
  }
  // Same blocking rule as reduce_sum_f32, capped at the array's capacity.
  int64_t chunks = std::max(d->slots, (n + kTargetChunkNA - 1) / kTargetChunkNA);
  chunks = std::min(chunks, std::max<int64_t>(1, n / kMinChunkNA));
  chunks = std::min(chunks, kNoAllocMaxBlocks);
  const int64_t chunk_len = ((n + chunks - 1) / chunks + 3) / 4 * 4;
  chunks = (n + chunk_len - 1) / chunk_len;
  unsigned* ticket = reinterpret_cast<unsigned*>(d->scratch);
  float* partials = reinterpret_cast<float*>(d->scratch + kTicketBytes);
  if (chunks > 1) {
    // The array keeps whatever the last call left; the ticket must start at 0.
    e = cudaMemsetAsync(ticket, 0, sizeof(unsigned), s);
    if (e != cudaSuccess) return record_cuda_error(e);
  }
  {  // debug builds: the call's buffers and the array (a no-op otherwise)
    const void* rp[3] = {x, out, d->scratch};
    const size_t rb[3] = {(size_t)n * sizeof(float), sizeof(float), kScratchBytes};
    e = dbg_register_ranges(s, rp, rb, 3);
    if (e != cudaSuccess) return record_cuda_error(e);
  }
  ContigParams p{x, n, chunk_len, (int32_t)chunks, out, partials, ticket, kEpiNone};
  launch_pdl(k_reduce_contig<16, OpSum>, dim3((unsigned)chunks), kThreads, 0, s, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e);
  count_launch();
  return LIBREDUCE_OK;
}
