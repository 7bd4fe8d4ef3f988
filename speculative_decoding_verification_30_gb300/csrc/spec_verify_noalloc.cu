// spec_verify_noalloc: spec_verify with its workspace taken from a fixed array in
// the library's own device memory, for callers that cannot allocate device memory
// (see include/spec_verify.h). This file only supplies the scratch and forwards to
// spec_verify; the kernels and their arguments are unchanged.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/spec_verify.h"

namespace {

// The scratch. Zero-initialised when the module loads; every spec_verify call
// leaves its workspace zero-filled again, so it is zero at the start of each call.
static __device__ __align__(256) unsigned char sv_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];

// Device address of the scratch on the current device, looked up once per device
// (the lookup may load the module on that device).
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  if (cudaGetSymbolAddress(&p, sv_noalloc_scratch) != cudaSuccess) return nullptr;
  g_scratch_ptr[dev].store(p, std::memory_order_release);
  return p;
}

}  // namespace

extern "C" sv_status spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                                         sv_dtype dtype, const int32_t* draft_tokens,
                                         const float* temperature, const int32_t* top_k,
                                         const float* top_p, uint64_t philox_seed,
                                         uint64_t philox_offset, int B, int K, int V,
                                         int32_t* out_tokens, int32_t* out_n_accepted,
                                         void* stream) {
  if (B < 1 || B > 65535 || K < 1 || K > 16) return SV_ERR_SHAPE;
  if (spec_verify_workspace_bytes(B, K) > SV_NOALLOC_SCRATCH_BYTES) return SV_ERR_SCRATCH;
  void* scratch = scratch_on_current_device();
  if (!scratch) return SV_ERR_CUDA;
  const sv_status s =
      spec_verify(target_logits, draft_logits, dtype, draft_tokens, temperature, top_k, top_p,
                  philox_seed, philox_offset, B, K, V, out_tokens, out_n_accepted, scratch,
                  SV_NOALLOC_SCRATCH_BYTES, stream);
  if (s != SV_OK) {
    // A failed launch can leave kernels queued before it (greedy_kernel writes its
    // per-row slots first) with the scratch not zeroed again. A caller workspace can
    // be cleared by its owner; this one is private, so clear the part the call could
    // have used, in stream order after whatever was queued (no allocation).
    if (cudaMemsetAsync(scratch, 0, spec_verify_workspace_bytes(B, K),
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return SV_ERR_CUDA;
  }
  return s;
}
