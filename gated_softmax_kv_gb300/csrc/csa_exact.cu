// Exact-mode forward kernel of the CSA/HCA fused Compressor for sm_103a
// (csa_compress_fwd_exact, windows of W <= 8 slots; the exact-mode backward
// is the bitwise kernel of csa_bwd_bitwise.cu).
//
// cuDNN-frontend "CSA Fused Compressor", sections "Semantics" and "Numerics":
// the same operation as the default forward, computed in the eager order of
// an fp32 reference so that out carries its bits:
//   z_k = score_k + ape_k, m = max z, e_k = exp(z_k - m) correctly rounded,
//   den = sum e (slot order), p_k = e_k / den (IEEE),
//   out = sum_k RN(p_k kv_k) (slot order), one bf16 rounding.
//
// The correctly rounded exp costs some 40 instructions a lane where the
// default kernels spend two, so this kernel is bound by instruction issue,
// not by HBM. It is shaped for that: a thread owns one column pair of one
// row at a time (4-byte accesses, still one coalesced 128-byte request per
// warp and slot), runs the pair through the two-lane fp32 instructions, keeps
// its APE columns in registers for the whole launch and leaves the registers
// for more resident warps, and the unrolled body of a row stays small enough
// for the instruction caches.
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_bwd_common.cuh"  // kGroupingSms
#include "csa_device.cuh"
#include "csa_exp_cr.cuh"
#include "csa_internal.h"

namespace csa {

namespace {

constexpr int kExactThreads = 256;
// resident CTAs per SM the register allocation is sized for
#ifndef CSA_EXACT_FWD_MIN_BLOCKS
#define CSA_EXACT_FWD_MIN_BLOCKS 3
#endif

__device__ __forceinline__ uint32_t ld_stream4(const uint16_t* p) {
  return __ldcs(reinterpret_cast<const unsigned int*>(p));
}
__device__ __forceinline__ void st_stream4(uint16_t* p, uint32_t v) {
  __stcs(reinterpret_cast<unsigned int*>(p), v);
}
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(bf16_lo(w), bf16_hi(w));
}

// The softmax weights of one column pair over a window: p[k] = e_k / den.
template <int W>
__device__ __forceinline__ void exact_weights(float2 (&z)[W], const float* tab) {
  float2 m = z[0];
#pragma unroll
  for (int k = 1; k < W; ++k) m = make_float2(max_nan(m.x, z[k].x), max_nan(m.y, z[k].y));
  float2 den = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int k = 0; k < W; ++k) {
    z[k] = exp_cr2(sub2_rn(z[k], m), tab);
    den = add2_rn(den, z[k]);
  }
  const float2 nden = make_float2(-den.x, -den.y);
  const float2 y = make_float2(__frcp_rn(den.x), __frcp_rn(den.y));
#pragma unroll
  for (int k = 0; k < W; ++k) z[k] = div2_cr(z[k], den, nden, y);
}

// Forward: blockDim = (TX column pairs, TY rows); rows strided by the grid.
// D > 0 fixes head_dim at compile time (slot offsets become immediates);
// D == 0 reads it from the problem.
template <int R, int COFF, int D>
__global__ void __launch_bounds__(kExactThreads, CSA_EXACT_FWD_MIN_BLOCKS)
fwd_exact_kernel(const FwdParams f) {
  grid_dependency_wait();
  allow_dependent_launch();
  constexpr int W = COFF * R;
  using S = Slot<R, COFF>;
  const Problem& p = f.p;
  const int d = D > 0 ? D : p.d;
  __shared__ float tab[2 * kExpTableSize];
  exp_cr_table(tab);
  __syncthreads();
  const int jp = blockIdx.x * blockDim.x + threadIdx.x;
  if (jp >= d / 2) return;  // no barrier below
  const int j0 = 2 * jp;
  const int64_t ld = (int64_t)COFF * d;
  float2 a[W];
#pragma unroll
  for (int k = 0; k < W; ++k)
    a[k] = __ldg(reinterpret_cast<const float2*>(p.ape + (int64_t)S::ape_row(k) * ld +
                                                 S::half(k) * d + j0));

  const int64_t true_rows = __ldg(p.cuc + p.nseq);
  const int64_t stride = (int64_t)gridDim.y * blockDim.y;
  int hint = 0;
  for (int64_t b = (int64_t)blockIdx.y * blockDim.y + threadIdx.y; b < p.C; b += stride) {
    const RowInfo ri = row_info_from(p.cu, p.cuc, p.nseq, b, true_rows, R, hint);
    uint16_t* dst = f.out + b * d + j0;
    if (!row_in_bounds<R, COFF>(ri, p.T)) {  // violated preconditions: NaN, no access
      st_stream4(dst, 0x7FC07FC0u);
      continue;
    }
    const int64_t rowoff = ri.base * ld + j0;
    uint32_t kvw[W], scw[W];
#pragma unroll
    for (int k = 0; k < W; ++k) {
      if (S::masked(ri.first, k)) {  // kv = 0, score = -inf
        kvw[k] = 0u;
        scw[k] = kNegInfBf16x2;
      } else {
        const int64_t off = rowoff + S::tok(0, k) * ld + S::half(k) * d;
        kvw[k] = ld_stream4(p.kv + off);
        scw[k] = ld_stream4(p.score + off);
      }
    }
    float2 z[W];
#pragma unroll
    for (int k = 0; k < W; ++k) z[k] = add2_rn(bf16x2_to_float2(scw[k]), a[k]);
    exact_weights<W>(z, tab);
    // out = sum_k RN(p_k kv_k); the products stay scalar (they feed a sum)
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < W; ++k)
      acc = add2_rn(acc, make_float2(__fmul_rn(z[k].x, bf16_lo(kvw[k])),
                                     __fmul_rn(z[k].y, bf16_hi(kvw[k]))));
    st_stream4(dst, pack_bf16x2(acc.x, acc.y));
  }
}

struct ExactShape {
  int tx, ty, tiles;
};

ExactShape exact_shape(int d) {
  ExactShape s;
  const int npair = d / 2;
  s.tx = npair <= 128 ? npair : 128;
  s.ty = kExactThreads / s.tx > 0 ? kExactThreads / s.tx : 1;
  s.tiles = (npair + s.tx - 1) / s.tx;
  return s;
}

// Row blocks per column tile: every resident CTA slot of the GPU, at most
// one per TY rows.
int64_t exact_rows_grid(const void* kern, const ExactShape& s, size_t smem, int64_t rows) {
  const int occ = occupancy(kern, s.tx * s.ty, smem);
  int64_t gy = (int64_t)kGroupingSms * occ / s.tiles;
  const int64_t row_blocks = (rows + s.ty - 1) / s.ty;
  if (gy > row_blocks) gy = row_blocks;
  if (gy < 1) gy = 1;
  if (gy > 65535) gy = 65535;
  return gy;
}

template <int R, int COFF, int D>
cudaError_t launch_fwd_exact_d(const FwdParams& f, cudaStream_t stream) {
  const ExactShape s = exact_shape(f.p.d);
  auto kern = fwd_exact_kernel<R, COFF, D>;
  const int64_t gy = exact_rows_grid(reinterpret_cast<const void*>(kern), s, 0, f.p.C);
  return launch_dependent(kern, dim3(s.tiles, (unsigned)gy), dim3(s.tx, s.ty), 0, stream, f);
}

template <int R, int COFF>
cudaError_t launch_fwd_exact_rc(const FwdParams& f, cudaStream_t stream) {
  if (f.p.d == 512) return launch_fwd_exact_d<R, COFF, 512>(f, stream);
  if (f.p.d == 128) return launch_fwd_exact_d<R, COFF, 128>(f, stream);
  return launch_fwd_exact_d<R, COFF, 0>(f, stream);
}

#define CSA_EXACT_DISPATCH(FN, ...)                 \
  switch (p.ratio * 4 + p.coff) {                   \
    case 2 * 4 + 1: return FN<2, 1>(__VA_ARGS__);   \
    case 2 * 4 + 2: return FN<2, 2>(__VA_ARGS__);   \
    case 4 * 4 + 1: return FN<4, 1>(__VA_ARGS__);   \
    case 4 * 4 + 2: return FN<4, 2>(__VA_ARGS__);   \
    case 8 * 4 + 1: return FN<8, 1>(__VA_ARGS__);   \
    default: return cudaErrorInvalidValue;          \
  }

}  // namespace

cudaError_t launch_fwd_exact(const FwdParams& f, cudaStream_t stream) {
  const Problem& p = f.p;
  if (p.C == 0) return cudaSuccess;
  CSA_EXACT_DISPATCH(launch_fwd_exact_rc, f, stream)
}

}  // namespace csa
