// csa_check_segments (declared in include/csa_compress.h): the device-side
// preconditions of the segment arrays that the compute calls trust
// (cuDNN-frontend "CSA Fused Compressor", sections "Semantics" and "Support
// surface"), checked on request by one kernel that ORs a bit per kind of
// violation into a caller-owned device word.
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_compress.h"
#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

namespace {

// One thread per segment (grid-strided); OR is commutative, so the word is
// the same whatever order the threads run in.
__global__ void check_segments_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ cuc,
                                      int32_t nseq, int64_t T, int64_t C, int32_t ratio,
                                      int32_t* __restrict__ violations) {
  grid_dependency_wait();
  allow_dependent_launch();
  int32_t bits = 0;
  for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < nseq;
       s += (int64_t)gridDim.x * blockDim.x) {
    const int64_t a = __ldg(cu + s), b = __ldg(cu + s + 1);
    const int64_t ca = __ldg(cuc + s), cb = __ldg(cuc + s + 1);
    if (s == 0 && (a != 0 || ca != 0)) bits |= CSA_SEG_BAD_START;
    if (b < a)
      bits |= CSA_SEG_DECREASING;
    else if (cb - ca != (b - a) / ratio)
      bits |= CSA_SEG_BAD_COMP;
    if (s == nseq - 1) {
      if (b > T) bits |= CSA_SEG_PAST_END;
      if (cb > C) bits |= CSA_SEG_OVER_CAPACITY;
    }
  }
  if (bits) atomicOr(violations, bits);
}

cudaError_t launch_check_segments(const int32_t* cu, const int32_t* cuc, int32_t nseq, int64_t T,
                                  int64_t C, int32_t ratio, int32_t* violations,
                                  cudaStream_t stream) {
  const int threads = 256;
  int64_t blocks = ((int64_t)nseq + threads - 1) / threads;
  if (blocks > 1024) blocks = 1024;
  return launch_dependent(check_segments_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                          cu, cuc, nseq, T, C, ratio, violations);
}

}  // namespace

}  // namespace csa

extern "C" csa_status_t csa_check_segments(const int32_t* cu_seqlens,
                                           const int32_t* cu_seqlens_comp, int32_t num_seqs,
                                           int64_t total_tokens, int64_t capacity, int32_t ratio,
                                           int32_t* violations, cudaStream_t stream) {
  if (!csa::supported(ratio, 1)) return CSA_ERR_UNSUPPORTED;
  if (num_seqs < 1 || total_tokens < 0 || capacity < 0) return CSA_ERR_RANGE;
  if (!cu_seqlens || !cu_seqlens_comp || !violations) return CSA_ERR_NULL;
  const uintptr_t a = reinterpret_cast<uintptr_t>(cu_seqlens) |
                      reinterpret_cast<uintptr_t>(cu_seqlens_comp) |
                      reinterpret_cast<uintptr_t>(violations);
  if (a % 4 != 0) return CSA_ERR_ALIGN;
  const cudaError_t e = csa::launch_check_segments(cu_seqlens, cu_seqlens_comp, num_seqs,
                                                   total_tokens, capacity, ratio, violations,
                                                   stream);
  return e == cudaSuccess ? CSA_OK : csa::record_cuda_error(e);
}
