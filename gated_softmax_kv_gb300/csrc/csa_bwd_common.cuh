// Device code shared by the two backward kernel shapes (csa_bwd.cu and
// csa_bwd_long.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

// The backward kernels' row-group count (the number of dAPE partials) is
// sized for this many SMs, not for the device's own count, so the grouping
// and with it dape's bits depend on the problem alone on every sm_103a part
// (152 is GB300's count; on a part with fewer SMs the few extra CTAs queue).
constexpr int kGroupingSms = 152;

// Zeros for the positions no row reads that belong to nobody's window:
// segments shorter than the ratio and tokens >= cu_seqlens[num_seqs].
// Spread over every CTA of the launch.
__device__ __forceinline__ void zero_orphans(const BwdParams& bp, int ratio) {
  const Problem& p = bp.p;
  const int64_t ld = (int64_t)p.coff * p.d;
  const int64_t vpt = ld / kVec;  // 16-byte vectors per token row
  const int nthr = blockDim.x * blockDim.y;
  const int tid = threadIdx.y * blockDim.x + threadIdx.x;
  const int64_t fb = (int64_t)blockIdx.y * gridDim.x + blockIdx.x;
  const int64_t nb = (int64_t)gridDim.x * gridDim.y;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t s = fb; s < p.nseq; s += nb) {
    int64_t lo = __ldg(p.cu + s), hi = __ldg(p.cu + s + 1);
    if (hi - lo >= ratio || hi <= lo) continue;
    lo = lo < 0 ? 0 : lo;
    hi = hi > p.T ? p.T : hi;
    for (int64_t v = lo * vpt + tid; v < hi * vpt; v += nthr) {
      st_stream(bp.dkv + v * kVec, zero);
      st_stream(bp.dscore + v * kVec, zero);
    }
  }
  int64_t end = __ldg(p.cu + p.nseq);
  end = end < 0 ? 0 : (end > p.T ? p.T : end);
  for (int64_t v = end * vpt + fb * nthr + tid; v < p.T * vpt; v += nb * nthr) {
    st_stream(bp.dkv + v * kVec, zero);
    st_stream(bp.dscore + v * kVec, zero);
  }
}

}  // namespace csa
