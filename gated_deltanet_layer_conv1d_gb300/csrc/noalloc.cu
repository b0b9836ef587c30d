// noalloc.cu -- gdn_prefill_chunked_noalloc: the chunked prefill for callers that cannot
// allocate device memory when they prefill (an engine that reserved almost all of HBM for
// its own pools at start-up, or a plug-in whose host runtime owns every allocation).  The
// workspace the chunked prefill needs comes from a fixed array in the library's own device
// memory instead of from the caller; the call itself allocates nothing.
#include <atomic>

#include "kernels.h"

namespace gdn {
namespace {

constexpr size_t kScratchBytes = GDN_NOALLOC_SCRATCH_BYTES;

// The scratch: one array per device that loads the library, kept until the process exits.
// Host code must not use the name as a device address; it looks the address up below.
// This file's module holds no kernel, so under CUDA's lazy module loading (the default) the
// array is reserved when the address is first looked up, not when the library loads: the
// first call per device (a call with n = 0 does only that) must come before the caller
// reserves the rest of the device's memory.
static __device__ __align__(256) unsigned char g_prefill_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<uintptr_t> g_scratch_addr[kMaxDevices];

// Device address of the scratch on the current device, looked up once per device and kept
// for the life of the process (a cudaDeviceReset would leave it stale).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  uintptr_t a = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (a == 0) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_prefill_scratch);
    if (e != cudaSuccess) return e;
    a = reinterpret_cast<uintptr_t>(ptr);
    g_scratch_addr[dev].store(a, std::memory_order_release);
  }
  *out = reinterpret_cast<void*>(a);
  return cudaSuccess;
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_prefill_chunked_noalloc(
    const gdn_dims* dims, const gdn_weights* weights, const gdn_inputs* inputs, int32_t n,
    const int32_t* cu_seqlens_dev, int32_t total_tokens, int32_t max_seqlen, int32_t chunk,
    const uint64_t* h_state_ptrs_dev, void* conv_pool, int32_t n_slots,
    const int32_t* slots_dev, void* y, float* core_out, int32_t* status_dev,
    gdn_stream_t stream) {
  if (!dims) return GDN_ERR_NULL_POINTER;
  const size_t need = gdn_prefill_workspace_bytes(dims, n, total_tokens, max_seqlen, chunk);
  if (need > gdn::kScratchBytes) return GDN_ERR_SCRATCH_TOO_SMALL;
  // The look-up runs on every call, n = 0 included, so that a call with nothing to do is
  // the set-up call: it reserves the array (lazy module loading) and caches its address.
  void* scratch = nullptr;
  if (gdn::scratch_address(&scratch) != cudaSuccess) return GDN_ERR_CUDA;
  return gdn_prefill_chunked(dims, weights, inputs, n, cu_seqlens_dev, total_tokens, max_seqlen,
                             chunk, h_state_ptrs_dev, conv_pool, n_slots, slots_dev, y,
                             core_out, scratch, need, status_dev, stream);
}
