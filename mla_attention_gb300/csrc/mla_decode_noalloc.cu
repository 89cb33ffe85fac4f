// mla_decode_noalloc: paged decode for callers that cannot allocate device memory.
//
// mla_decode needs a caller-owned workspace for its split-K partial results.
// Some callers cannot provide one because they cannot call cudaMalloc (or any
// allocator) where they run attention: plug-ins that a host framework hands
// only the input and output buffers (the framework owns every device
// allocation), processes that forbid device allocation after start-up
// (real-time or certified deployments), and callers whose memory comes from a
// pool they cannot grow from inside this call.  This entry point serves them:
// the caller passes inputs and outputs only, and the scratch lives in a
// file-scope __device__ array of this library, kNoAllocScratchBytes long
// (50,446,848 bytes, about 48.1 MiB).  Every GPU that loads the library holds that array until
// the process exits.  No cudaMalloc, cudaFree or allocating routine is called.
//
// Set-up: the first call on a device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress and caches it; make that
// first call before any stream capture.  All calls share the array and it
// keeps the last call's contents; each call clears the status word it needs
// at zero.  Calls that overlap on the GPU (other streams, or before the
// previous call finished) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kNoAllocMaxBatch = 4096;   // requests per call
constexpr int kNoAllocMaxRows = 24576;   // (requests + CTA pairs) x heads partial rows
constexpr size_t round256(size_t x) { return (x + 255) / 256 * 256; }
constexpr size_t kNoAllocScratchBytes = kWsHeader + round256(sizeof(int32_t) * (kNoAllocMaxBatch + 1)) +
                                        round256(sizeof(float) * (size_t)kNoAllocMaxRows) +
                                        sizeof(float) * (size_t)kNoAllocMaxRows * kLatent;

// In host code this name is a host-side stand-in, not a device address: the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status mla_decode_noalloc(const void* q, const void* kv_cache, int64_t num_pages, int page_size,
                                         const int32_t* block_table, int max_pages, const int32_t* lens, int B,
                                         int H, float scale, int num_splits, void* out, float* lse, void* stream) {
  if (B < 0 || B > kNoAllocMaxBatch)
    return set_last_error(MLA_ERR_INVALID_ARG, "mla_decode_noalloc: B must be in [0, 4096]");
  if (H < 1 || num_splits < 0) return set_last_error(MLA_ERR_INVALID_ARG, "mla_decode_noalloc: H >= 1, num_splits >= 0");
  int pairs = num_splits > 0 ? num_splits : device_sm_count() / 2;
  if (pairs < 1) pairs = 1;
  if ((int64_t)(B + pairs) * H > kNoAllocMaxRows)
    return set_last_error(MLA_ERR_INVALID_ARG,
                          "mla_decode_noalloc: (B + CTA pairs) * H must be <= 24576 (use fewer splits or requests)");
  if (mla_decode_workspace_size(B, H, num_splits) > kNoAllocScratchBytes)
    return set_last_error(MLA_ERR_INVALID_ARG, "mla_decode_noalloc: the call needs more scratch than the fixed array");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_last_error(MLA_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return set_last_error(MLA_ERR_UNSUPPORTED, "mla_decode_noalloc: device index >= 64");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
      if (e != cudaSuccess || !ptr) return set_last_error(MLA_ERR_CUDA, "mla_decode_noalloc: cudaGetSymbolAddress failed");
      g_scratch_ptr[dev] = ptr;
    }
    scratch = g_scratch_ptr[dev];
  }
  // the device status word at the head of the scratch must start at zero
  e = cudaMemsetAsync(scratch, 0, sizeof(uint32_t), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return set_last_error(MLA_ERR_CUDA, cudaGetErrorString(e));
  return mla_decode(q, kv_cache, num_pages, page_size, block_table, max_pages, lens, B, H, scale, num_splits, out,
                    lse, scratch, kNoAllocScratchBytes, stream);
}
