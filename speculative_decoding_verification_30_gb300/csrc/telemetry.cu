// telemetry.cu -- acceptance telemetry for the verify step (sm_103a).
//
// The pages' main operational signal for speculative decoding is the acceptance
// rate and the draft depth it supports ("Speculative decoding: draft models,
// VRAM economics, 3x", section on acceptance rates and draft length; "MTPLX",
// section on the tune command). spec_accept_histogram counts, over the sequences
// of one or more verify calls, how many drafted tokens were accepted, so that the
// host can estimate per-position acceptance rates and choose a depth without
// copying every call's outputs back.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spec_verify.h"

namespace sv {

// hist[n] += #{b : n_accepted[b] == n} for n in [0, K]; hist[K + 1] counts data
// errors (n = -1) and any value outside [0, K].
__global__ void accept_hist_kernel(const int32_t* n_accepted, int B, int K, unsigned long long* hist) {
  extern __shared__ unsigned int bins[];
  for (int i = threadIdx.x; i < K + 2; i += blockDim.x) bins[i] = 0u;
  __syncthreads();
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
    const int v = n_accepted[b];
    atomicAdd(&bins[(v >= 0 && v <= K) ? v : K + 1], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < K + 2; i += blockDim.x)
    if (bins[i]) atomicAdd(&hist[i], (unsigned long long)bins[i]);
}

}  // namespace sv

extern "C" sv_status spec_accept_histogram(const int32_t* n_accepted, int B, int K,
                                           unsigned long long* hist, void* stream) {
  if (B < 1 || K < 1 || K > 16) return SV_ERR_SHAPE;
  if (!n_accepted || !hist) return SV_ERR_NULL;
  if ((uintptr_t)n_accepted % 4 || (uintptr_t)hist % 8) return SV_ERR_ALIGN;
  const int threads = 256;
  int grid = (B + threads - 1) / threads;
  if (grid > 64) grid = 64;
  sv::accept_hist_kernel<<<grid, threads, (size_t)(K + 2) * sizeof(unsigned int),
                           static_cast<cudaStream_t>(stream)>>>(n_accepted, B, K, hist);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
