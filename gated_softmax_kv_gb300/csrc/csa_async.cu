// The device fault word of the producer/consumer kernels: bounded waits that
// give up OR a flag into it (see csa_async.cuh); the host reads and clears it
// through csa_read_device_faults.
#include <cuda.h>
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

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace

cudaError_t encode_bf16_rows(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                             uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
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
