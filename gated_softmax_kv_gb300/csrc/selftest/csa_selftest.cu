// Test hooks for device helpers of the Compressor kernels (not part of the
// C ABI in include/csa_compress.h): built into libcsa_selftest.so, loaded
// only by the GPU tests.
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_device.cuh"

namespace {

__global__ void softmax_exp_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    y[i] = csa::softmax_exp(x[i]);
}

__global__ void softmax_exp_fast_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    y[i] = csa::softmax_exp_fast(x[i]);
}

__global__ void div_kernel(const float* __restrict__ a, const float* __restrict__ b,
                           float* __restrict__ q, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    q[i] = csa::div_rn_by_rcp(a[i], b[i], __frcp_rn(b[i]));
}

}  // namespace

extern "C" int32_t csa_selftest_div(const float* a, const float* b, float* q, int64_t n,
                                    cudaStream_t stream) {
  if (n <= 0) return 0;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  div_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a, b, q, n);
  return (int32_t)cudaGetLastError();
}

extern "C" int32_t csa_selftest_softmax_exp_fast(const float* x, float* y, int64_t n,
                                                 cudaStream_t stream) {
  if (n <= 0) return 0;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  softmax_exp_fast_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, y, n);
  return (int32_t)cudaGetLastError();
}

extern "C" int32_t csa_selftest_softmax_exp(const float* x, float* y, int64_t n,
                                            cudaStream_t stream) {
  if (n <= 0) return 0;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  softmax_exp_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, y, n);
  return (int32_t)cudaGetLastError();
}
