// Internal interface between the C ABI (csa_api.cu, csa_noalloc.cu) and the
// kernel translation units (csa_fwd.cu, csa_fwd_long.cu, csa_bwd.cu,
// csa_bwd_long.cu, csa_fwd_bitwise.cu, csa_bwd_bitwise.cu). Not installed,
// not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace csa {

// Launches `kernel` on `stream` with programmatic stream serialization (the
// kernel's launch may overlap the previous kernel's tail; the kernel waits for
// that grid with griddepcontrol.wait before touching memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
#ifdef CSA_NO_PDL
  cfg.numAttrs = 0;  // plain stream order (comparison builds)
#else
  cfg.numAttrs = 1;
#endif
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// One Compressor call after host validation. Pointers are device pointers;
// bf16 tensors travel as raw 16-bit patterns.
struct Problem {
  const uint16_t* kv;      // [T, coff*d]
  const uint16_t* score;   // [T, coff*d]
  const float* ape;        // [ratio, coff*d]
  const int32_t* cu;       // [nseq + 1]
  const int32_t* cuc;      // [nseq + 1]
  int32_t nseq;
  int32_t ratio;
  int32_t coff;
  int32_t d;               // head_dim
  int64_t T;               // total_tokens
  int64_t C;               // capacity
  bool exact;              // exact mode: correctly rounded exp, IEEE division, eager order
};

struct FwdParams {
  Problem p;
  uint16_t* out;           // [C, d]
};

struct BwdParams {
  Problem p;
  const uint16_t* grad_out;  // [C, d]
  uint16_t* dkv;             // [T, coff*d]
  uint16_t* dscore;          // [T, coff*d]
  float* partial;            // [groups, ratio * coff * d] dape partials
  int32_t groups;            // row groups = number of partials
};

// Launch shape of the backward: how many dape partials it writes.
struct BwdShape {
  dim3 grid;
  dim3 block;
  size_t smem;
  int32_t groups;
};

bool supported(int ratio, int coff);

cudaError_t launch_fwd(const FwdParams& f, cudaStream_t stream);

cudaError_t plan_bwd(const Problem& p, BwdShape* shape);
cudaError_t launch_bwd(const BwdParams& b, const BwdShape& shape, cudaStream_t stream);
// Windows of 16 slots and more (csa_fwd_long.cu, csa_bwd_long.cu).
cudaError_t launch_fwd_long(const FwdParams& f, cudaStream_t stream);
cudaError_t plan_bwd_long(const Problem& p, BwdShape* shape);
cudaError_t launch_bwd_long(const BwdParams& b, const BwdShape& shape, cudaStream_t stream);
// The exact-mode (bitwise) forward, windows of at most 8 slots
// (csa_fwd_bitwise.cu).
cudaError_t launch_fwd_bitwise(const FwdParams& f, cudaStream_t stream);
// The bitwise backward for windows of at most 8 slots (csa_bwd_bitwise.cu).
cudaError_t plan_bwd_bitwise(const Problem& p, BwdShape* shape);
cudaError_t launch_bwd_bitwise(const BwdParams& b, const BwdShape& shape, cudaStream_t stream);
cudaError_t launch_dape_reduce(const float* partial, int32_t groups, int64_t n, float* dape,
                               cudaStream_t stream);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();
// Resident CTAs per SM of a kernel (at least 1).
int occupancy(const void* kernel, int threads, size_t smem);
// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device); the attribute is per device.
cudaError_t allow_dynamic_smem(const void* kernel, int bytes);

}  // namespace csa

#include "csa_compress.h"

namespace csa {

// Backward argument checks shared with the allocation-free entry point, and
// the per-thread record behind csa_last_cuda_error() (csa_api.cu).
csa_status_t check_bwd_args(const void* kv, const void* score, const float* ape, const int32_t* cu,
                            const int32_t* cuc, int32_t num_seqs, int64_t total_tokens,
                            int64_t capacity, int32_t ratio, int32_t coff, int32_t head_dim,
                            const void* grad_out, const void* dkv, const void* dscore,
                            const float* dape);
csa_status_t record_cuda_error(cudaError_t e);

// The unique id of the CUDA context current on this thread (the driver's
// context id, unique for the life of the process), creating the device's
// primary context first if none is current. Host-side caches of per-context
// objects (device symbol addresses, memory pools) are keyed by it, so that
// a context destroyed and created again (cudaDeviceReset) is never served a
// stale handle.
cudaError_t current_context_id(unsigned long long* id);

}  // namespace csa
