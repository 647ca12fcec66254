// The device fault word of the producer/consumer kernels: bounded waits that
// give up OR a flag into it (see csa_async.cuh); the host reads and clears it
// through csa_read_device_faults.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "csa_compress.h"
#include "csa_internal.h"

namespace {

__device__ unsigned int g_faults = 0u;

}  // namespace

namespace csa {

cudaError_t device_fault_word(unsigned int** out) {
  static std::mutex mu;
  static unsigned int* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_faults);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<unsigned int*>(p);
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace csa

extern "C" csa_status_t csa_read_device_faults(int32_t* flags) {
  if (!flags) return CSA_ERR_NULL;
  unsigned int v = 0u;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_faults, sizeof v);
  if (e != cudaSuccess) return csa::record_cuda_error(e);
  const unsigned int zero = 0u;
  e = cudaMemcpyToSymbol(g_faults, &zero, sizeof zero);
  if (e != cudaSuccess) return csa::record_cuda_error(e);
  *flags = (int32_t)v;
  return CSA_OK;
}
