// csa_compress_bwd_noalloc: the backward without any device allocation.
//
// For callers that cannot allocate device memory while the backward runs
// (all device memory handed to their own allocator at start-up, or a
// time-critical loop that must stay out of the CUDA allocator). The
// backward's only scratch -- the per-row-group dape partials -- lives here in
// one file-scope device array instead of the stream-ordered pool that
// csa_compress_bwd uses. Kernels, launch shape and results are those of
// csa_compress_bwd.
//
// In host code `g_dape_scratch` names a host-side stand-in, not device
// memory: the kernels get the device address that cudaGetSymbolAddress
// returns, looked up on the first call in each CUDA context of a device (with
// that device current) and cached under the context's unique id, so that a
// context destroyed and created again (cudaDeviceReset) makes the next call
// look the address up again instead of launching with a stale one. Every
// call shares the array; calls whose kernels overlap on the GPU race on it.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "csa_compress.h"
#include "csa_internal.h"

namespace {

constexpr int64_t kScratchFloats = CSA_NOALLOC_SCRATCH_FLOATS;  // 16 MiB per device
static_assert(kScratchFloats == 4 * 1024 * 1024, "scratch size is part of the documented ABI");

static __device__ __align__(256) float g_dape_scratch[kScratchFloats];

// Device address of g_dape_scratch in the current context, looked up once per
// (device, context).
cudaError_t scratch_address(float** out) {
  static std::mutex mu;
  struct Entry {
    unsigned long long ctx;
    float* addr;
  };
  static Entry cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  unsigned long long ctx = 0;
  e = csa::current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev].addr || cache[dev].ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dape_scratch);
    if (e != cudaSuccess) return e;
    cache[dev].addr = static_cast<float*>(p);
    cache[dev].ctx = ctx;
  }
  *out = cache[dev].addr;
  return cudaSuccess;
}

}  // namespace

extern "C" csa_status_t csa_compress_bwd_noalloc(
    const void* kv, const void* score, const float* ape, const int32_t* cu_seqlens,
    const int32_t* cu_seqlens_comp, int32_t num_seqs, int64_t total_tokens, int64_t capacity,
    int32_t ratio, int32_t coff, int32_t head_dim, const void* grad_out, void* dkv, void* dscore,
    float* dape, cudaStream_t stream) {
  csa_status_t st = csa::check_bwd_args(kv, score, ape, cu_seqlens, cu_seqlens_comp, num_seqs,
                                        total_tokens, capacity, ratio, coff, head_dim, grad_out,
                                        dkv, dscore, dape);
  if (st != CSA_OK) return st;

  csa::BwdParams b;
  b.p.kv = static_cast<const uint16_t*>(kv);
  b.p.score = static_cast<const uint16_t*>(score);
  b.p.ape = ape;
  b.p.cu = cu_seqlens;
  b.p.cuc = cu_seqlens_comp;
  b.p.nseq = num_seqs;
  b.p.ratio = ratio;
  b.p.coff = coff;
  b.p.d = head_dim;
  b.p.T = total_tokens;
  b.p.C = capacity;
  b.p.exact = false;
  b.grad_out = static_cast<const uint16_t*>(grad_out);
  b.dkv = static_cast<uint16_t*>(dkv);
  b.dscore = static_cast<uint16_t*>(dscore);

  csa::BwdShape shape;
  cudaError_t e = csa::plan_bwd(b.p, &shape);
  if (e != cudaSuccess) return csa::record_cuda_error(e);
  const int64_t n_ape = (int64_t)ratio * coff * head_dim;
  if (n_ape * shape.groups > kScratchFloats) return CSA_ERR_SCRATCH;

  float* scratch = nullptr;
  e = scratch_address(&scratch);
  if (e != cudaSuccess) return csa::record_cuda_error(e);
  // every partial the reduce reads is written by this call's backward kernel
  b.partial = scratch;
  b.groups = shape.groups;
  e = csa::launch_bwd(b, shape, stream);
  if (e == cudaSuccess) e = csa::launch_dape_reduce(b.partial, shape.groups, n_ape, dape, stream);
  if (e != cudaSuccess) return csa::record_cuda_error(e);
  return CSA_OK;
}
