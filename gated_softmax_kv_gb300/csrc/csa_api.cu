// C ABI of the CSA/HCA fused Compressor (declared in include/csa_compress.h).
//
// Host side only: argument validation (cuDNN-frontend "CSA Fused Compressor",
// section "Support surface"), kernel dispatch and the stream-ordered dape
// workspace. No call synchronises the host; no device memory is read here.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "csa_compress.h"
#include "csa_internal.h"

namespace {

thread_local int32_t g_last_cuda_error = 0;

csa_status_t cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int32_t)e;
  return CSA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shared checks of both directions. Pointers that index no element (an empty
// tensor) may be null.
csa_status_t validate(const void* kv, const void* score, const float* ape, const int32_t* cu,
                      const int32_t* cuc, int32_t num_seqs, int64_t total_tokens,
                      int64_t capacity, int32_t ratio, int32_t coff, int32_t head_dim) {
  if (!csa::supported(ratio, coff)) return CSA_ERR_UNSUPPORTED;
  if (head_dim < 8 || head_dim % 8 != 0) return CSA_ERR_UNSUPPORTED;
  if (num_seqs < 1 || total_tokens < 0 || capacity < 0) return CSA_ERR_RANGE;
  const int64_t lim = (int64_t)1 << 31;
  if (total_tokens > lim / ((int64_t)coff * head_dim)) return CSA_ERR_RANGE;
  if (total_tokens * coff * head_dim >= lim || capacity * (int64_t)head_dim >= lim)
    return CSA_ERR_RANGE;
  if (capacity > 0 && total_tokens < ratio) return CSA_ERR_RANGE;
  if (!cu || !cuc || !ape) return CSA_ERR_NULL;
  if (total_tokens > 0 && (!kv || !score)) return CSA_ERR_NULL;
  if (!aligned(cu, 4) || !aligned(cuc, 4)) return CSA_ERR_ALIGN;
  if (!aligned(kv, 16) || !aligned(score, 16) || !aligned(ape, 16)) return CSA_ERR_ALIGN;
  return CSA_OK;
}

csa::Problem make_problem(const void* kv, const void* score, const float* ape, const int32_t* cu,
                          const int32_t* cuc, int32_t num_seqs, int64_t total_tokens,
                          int64_t capacity, int32_t ratio, int32_t coff, int32_t head_dim) {
  csa::Problem p;
  p.kv = static_cast<const uint16_t*>(kv);
  p.score = static_cast<const uint16_t*>(score);
  p.ape = ape;
  p.cu = cu;
  p.cuc = cuc;
  p.nseq = num_seqs;
  p.ratio = ratio;
  p.coff = coff;
  p.d = head_dim;
  p.T = total_tokens;
  p.C = capacity;
  p.exact = false;
  return p;
}

// One pool per CUDA context for the dape partials. The release threshold
// keeps the memory cached between calls, so steady-state calls do not map
// new memory. The cache is keyed by the context id: after a device reset the
// next call creates a pool in the new context instead of using the old one.
cudaError_t workspace_pool(cudaMemPool_t* out) {
  static std::mutex mu;
  struct Entry {
    unsigned long long ctx;
    cudaMemPool_t pool;
  };
  static Entry pools[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  unsigned long long ctx = 0;
  e = csa::current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (!pools[dev].pool || pools[dev].ctx != ctx) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool;
    e = cudaMemPoolCreate(&pool, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = UINT64_MAX;
    e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return e;
    pools[dev].pool = pool;
    pools[dev].ctx = ctx;
  }
  *out = pools[dev].pool;
  return cudaSuccess;
}

// Exact mode (csa_compress_fwd_exact / csa_compress_bwd_exact): the
// small-window shapes only (coff * ratio <= 8).
bool exact_supported(int32_t ratio, int32_t coff) { return coff * ratio <= 8; }

csa_status_t fwd_call(const void* kv, const void* score, const float* ape, const int32_t* cu_seqlens,
                      const int32_t* cu_seqlens_comp, int32_t num_seqs, int64_t total_tokens,
                      int64_t capacity, int32_t ratio, int32_t coff, int32_t head_dim, void* out,
                      cudaStream_t stream, bool exact) {
  csa_status_t st = validate(kv, score, ape, cu_seqlens, cu_seqlens_comp, num_seqs, total_tokens,
                             capacity, ratio, coff, head_dim);
  if (st != CSA_OK) return st;
  if (exact && !exact_supported(ratio, coff)) return CSA_ERR_UNSUPPORTED;
  if (capacity > 0 && !out) return CSA_ERR_NULL;
  if (!aligned(out, 16)) return CSA_ERR_ALIGN;
  if (capacity == 0) return CSA_OK;
  csa::FwdParams f;
  f.p = make_problem(kv, score, ape, cu_seqlens, cu_seqlens_comp, num_seqs, total_tokens,
                     capacity, ratio, coff, head_dim);
  f.p.exact = exact;
  f.out = static_cast<uint16_t*>(out);
  cudaError_t e = csa::launch_fwd(f, stream);
  return e == cudaSuccess ? CSA_OK : cuda_fail(e);
}

csa_status_t bwd_call(const void* kv, const void* score, const float* ape, const int32_t* cu_seqlens,
                      const int32_t* cu_seqlens_comp, int32_t num_seqs, int64_t total_tokens,
                      int64_t capacity, int32_t ratio, int32_t coff, int32_t head_dim,
                      const void* grad_out, void* dkv, void* dscore, float* dape,
                      cudaStream_t stream, bool exact) {
  csa_status_t st = validate(kv, score, ape, cu_seqlens, cu_seqlens_comp, num_seqs, total_tokens,
                             capacity, ratio, coff, head_dim);
  if (st != CSA_OK) return st;
  if (exact && !exact_supported(ratio, coff)) return CSA_ERR_UNSUPPORTED;
  if ((capacity > 0 && !grad_out) || (total_tokens > 0 && (!dkv || !dscore)) || !dape)
    return CSA_ERR_NULL;
  if (!aligned(grad_out, 16) || !aligned(dkv, 16) || !aligned(dscore, 16) || !aligned(dape, 16))
    return CSA_ERR_ALIGN;

  csa::BwdParams b;
  b.p = make_problem(kv, score, ape, cu_seqlens, cu_seqlens_comp, num_seqs, total_tokens,
                     capacity, ratio, coff, head_dim);
  b.p.exact = exact;
  b.grad_out = static_cast<const uint16_t*>(grad_out);
  b.dkv = static_cast<uint16_t*>(dkv);
  b.dscore = static_cast<uint16_t*>(dscore);
  csa::BwdShape shape;
  cudaError_t e = csa::plan_bwd(b.p, &shape);
  if (e != cudaSuccess) return cuda_fail(e);
  b.groups = shape.groups;

  const int64_t n_ape = (int64_t)ratio * coff * head_dim;
  const size_t ws_bytes = sizeof(float) * (size_t)n_ape * (size_t)shape.groups;
  cudaMemPool_t pool;
  e = workspace_pool(&pool);
  if (e != cudaSuccess) return cuda_fail(e);
  void* ws = nullptr;
  e = cudaMallocFromPoolAsync(&ws, ws_bytes, pool, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  b.partial = static_cast<float*>(ws);
  e = csa::launch_bwd(b, shape, stream);
  if (e == cudaSuccess) e = csa::launch_dape_reduce(b.partial, shape.groups, n_ape, dape, stream);
  cudaError_t ef = cudaFreeAsync(ws, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  if (ef != cudaSuccess) return cuda_fail(ef);
  return CSA_OK;
}

}  // namespace

namespace csa {

// Argument checks of the backward, for the allocation-free entry point
// (csa_noalloc.cu); the same checks csa_compress_bwd makes.
csa_status_t check_bwd_args(const void* kv, const void* score, const float* ape, const int32_t* cu,
                            const int32_t* cuc, int32_t num_seqs, int64_t total_tokens,
                            int64_t capacity, int32_t ratio, int32_t coff, int32_t head_dim,
                            const void* grad_out, const void* dkv, const void* dscore,
                            const float* dape) {
  csa_status_t st = validate(kv, score, ape, cu, cuc, num_seqs, total_tokens, capacity, ratio,
                             coff, head_dim);
  if (st != CSA_OK) return st;
  if ((capacity > 0 && !grad_out) || (total_tokens > 0 && (!dkv || !dscore)) || !dape)
    return CSA_ERR_NULL;
  if (!aligned(grad_out, 16) || !aligned(dkv, 16) || !aligned(dscore, 16) || !aligned(dape, 16))
    return CSA_ERR_ALIGN;
  return CSA_OK;
}

csa_status_t record_cuda_error(cudaError_t e) { return cuda_fail(e); }

namespace {

// Driver entry points, looked up once through the runtime (no link against
// libcuda): cuCtxGetCurrent and cuCtxGetId.
typedef int (*CtxGetCurrentFn)(void** ctx);
typedef int (*CtxGetIdFn)(void* ctx, unsigned long long* id);

cudaError_t context_fns(CtxGetCurrentFn* cur, CtxGetIdFn* id) {
  static std::once_flag once;
  static CtxGetCurrentFn s_cur = nullptr;
  static CtxGetIdFn s_id = nullptr;
  static cudaError_t s_err = cudaSuccess;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    s_err = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q);
    if (s_err == cudaSuccess && q != cudaDriverEntryPointSuccess) s_err = cudaErrorNotSupported;
    if (s_err != cudaSuccess) return;
    s_cur = reinterpret_cast<CtxGetCurrentFn>(f);
    s_err = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q);
    if (s_err == cudaSuccess && q != cudaDriverEntryPointSuccess) s_err = cudaErrorNotSupported;
    if (s_err != cudaSuccess) return;
    s_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  *cur = s_cur;
  *id = s_id;
  return s_err;
}

}  // namespace

cudaError_t current_context_id(unsigned long long* out) {
  CtxGetCurrentFn cur;
  CtxGetIdFn getid;
  cudaError_t e = context_fns(&cur, &getid);
  if (e != cudaSuccess) return e;
  void* ctx = nullptr;
  if (cur(&ctx) != 0) return cudaErrorDeviceUninitialized;
  if (!ctx) {
    // no context current yet on this thread: let the runtime make the
    // current device's primary context current (no memory is allocated)
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (cur(&ctx) != 0 || !ctx) return cudaErrorDeviceUninitialized;
  }
  return getid(ctx, out) == 0 ? cudaSuccess : cudaErrorDeviceUninitialized;
}

}  // namespace csa

extern "C" {

csa_status_t csa_compress_fwd(const void* kv, const void* score, const float* ape,
                              const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                              int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                              int32_t ratio, int32_t coff, int32_t head_dim, void* out,
                              cudaStream_t stream) {
  return fwd_call(kv, score, ape, cu_seqlens, cu_seqlens_comp, num_seqs, total_tokens, capacity,
                  ratio, coff, head_dim, out, stream, false);
}

csa_status_t csa_compress_fwd_exact(const void* kv, const void* score, const float* ape,
                                    const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                                    int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                                    int32_t ratio, int32_t coff, int32_t head_dim, void* out,
                                    cudaStream_t stream) {
  return fwd_call(kv, score, ape, cu_seqlens, cu_seqlens_comp, num_seqs, total_tokens, capacity,
                  ratio, coff, head_dim, out, stream, true);
}

csa_status_t csa_compress_bwd(const void* kv, const void* score, const float* ape,
                              const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                              int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                              int32_t ratio, int32_t coff, int32_t head_dim,
                              const void* grad_out, void* dkv, void* dscore, float* dape,
                              cudaStream_t stream) {
  return bwd_call(kv, score, ape, cu_seqlens, cu_seqlens_comp, num_seqs, total_tokens, capacity,
                  ratio, coff, head_dim, grad_out, dkv, dscore, dape, stream, false);
}

csa_status_t csa_compress_bwd_exact(const void* kv, const void* score, const float* ape,
                                    const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                                    int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                                    int32_t ratio, int32_t coff, int32_t head_dim,
                                    const void* grad_out, void* dkv, void* dscore, float* dape,
                                    cudaStream_t stream) {
  return bwd_call(kv, score, ape, cu_seqlens, cu_seqlens_comp, num_seqs, total_tokens, capacity,
                  ratio, coff, head_dim, grad_out, dkv, dscore, dape, stream, true);
}

const char* csa_status_string(csa_status_t status) {
  switch (status) {
    case CSA_OK: return "ok";
    case CSA_ERR_NULL: return "a required pointer is null";
    case CSA_ERR_ALIGN: return "a base pointer is misaligned (16 bytes for tensors, 4 for segment arrays)";
    case CSA_ERR_UNSUPPORTED: return "ratio, coff or head_dim outside the supported envelope";
    case CSA_ERR_RANGE: return "a size is negative, overflows int32 flat offsets, or capacity > 0 with total_tokens < ratio";
    case CSA_ERR_CUDA: return "a CUDA runtime call failed";
    case CSA_ERR_SCRATCH: return "the backward needs more dape scratch than the no-allocation buffer holds (CSA_NOALLOC_SCRATCH_FLOATS)";
    default: return "unknown status";
  }
}

int32_t csa_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
