// Test hooks for device helpers of the Compressor kernels (not part of the
// C ABI in include/csa_compress.h): built into libcsa_selftest.so, loaded
// only by the GPU tests.
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_device.cuh"
#include "csa_exp_cr.cuh"

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

// The two-lane fp32 helpers one operation at a time (every result stored, so
// nothing can be fused), in the chains the kernels use (a product feeding a
// product, a difference feeding a product, an FMA, a scalar product feeding
// a two-lane sum or difference), and the scalar FMA.
__global__ void pair_ops_kernel(const float2* __restrict__ a, const float2* __restrict__ b,
                                const float2* __restrict__ c, float2* __restrict__ out,
                                int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float2 x = a[i], y = b[i], z = c[i];
    out[0 * n + i] = csa::add2_rn(x, y);
    out[1 * n + i] = csa::sub2_rn(x, z);
    out[2 * n + i] = csa::mul2_rn(y, z);
    out[3 * n + i] = csa::mul2_rn(csa::mul2_rn(x, y), z);
    out[4 * n + i] = csa::mul2_rn(csa::sub2_rn(x, y), z);
    out[5 * n + i] = csa::fma2_rn(x, y, z);
    out[6 * n + i] = make_float2(__fmaf_rn(x.x, y.x, z.x), __fmaf_rn(x.y, y.y, z.y));
    // scalar products feeding two-lane sums, as the exact mode chains them
    out[7 * n + i] = csa::add2_rn(x, make_float2(__fmul_rn(y.x, z.x), __fmul_rn(y.y, z.y)));
    out[8 * n + i] = csa::sub2_rn(make_float2(__fmul_rn(x.x, y.x), __fmul_rn(x.y, y.y)), z);
  }
}

__global__ void exp_cr2_kernel(const float2* __restrict__ x, float2* __restrict__ y, int64_t n) {
  __shared__ float tab[2 * csa::kExpTableSize];
  csa::exp_cr_table(tab);
  __syncthreads();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    y[i] = csa::exp_cr2(x[i], tab);
}

__global__ void div2_kernel(const float2* __restrict__ a, const float2* __restrict__ b,
                            float2* __restrict__ q, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float2 bb = b[i];
    q[i] = csa::div2_cr(a[i], bb, make_float2(-bb.x, -bb.y),
                        make_float2(__frcp_rn(bb.x), __frcp_rn(bb.y)));
  }
}

// Largest (|fast(t) - E| / E) 2^24 - kFastExpC1 |t| over every fp32 t whose
// encoding lies in [lo, hi] (negative numbers: -0 = 0x80000000 up to
// -kFastExpTMax), E = exp(t) in fp64 (within 2^-52 of the exact value), as
// the bits of a non-negative double combined with atomicMax (the order of
// non-negative doubles is that of their encodings); NaN or an infinite ratio
// records +inf.
__global__ void fast_exp_envelope_kernel(uint32_t lo, uint32_t hi,
                                         unsigned long long* __restrict__ worst) {
  double m = 0.0;
  const uint64_t n = (uint64_t)hi - lo + 1;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x) {
    const float t = __uint_as_float((uint32_t)(lo + i));
    const double e = exp((double)t);
    const double r = fabs((double)csa::softmax_exp_fast(t) - e) / e * 16777216.0 -
                     (double)csa::kFastExpC1 * fabs((double)t);
    m = (r == r) ? fmax(m, r) : __longlong_as_double(0x7ff0000000000000LL);
  }
  for (int o = 16; o > 0; o >>= 1) m = fmax(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(worst, (unsigned long long)__double_as_longlong(m));
}

}  // namespace

// The bitwise backward's envelope of softmax_exp_fast: the constants and the
// measured worst case over every fp32 t in [-kFastExpTMax, 0].
extern "C" void csa_selftest_fast_exp_constants(float* c0, float* c1, float* tmax) {
  *c0 = csa::kFastExpC0;
  *c1 = csa::kFastExpC1;
  *tmax = csa::kFastExpTMax;
}

// worst: one device unsigned long long, zeroed by the caller.
extern "C" int32_t csa_selftest_fast_exp_envelope(uint32_t lo_bits, uint32_t hi_bits,
                                                  unsigned long long* worst, cudaStream_t stream) {
  if (hi_bits < lo_bits) return 0;
  fast_exp_envelope_kernel<<<152 * 8, 256, 0, stream>>>(lo_bits, hi_bits, worst);
  return (int32_t)cudaGetLastError();
}

// div2_cr on n_pairs operand pairs (a[2i], a[2i + 1]) / (b[2i], b[2i + 1]).
extern "C" int32_t csa_selftest_div2(const float* a, const float* b, float* q, int64_t n_pairs,
                                     cudaStream_t stream) {
  if (n_pairs <= 0) return 0;
  int64_t blocks = (n_pairs + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  div2_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const float2*>(a),
                                                    reinterpret_cast<const float2*>(b),
                                                    reinterpret_cast<float2*>(q), n_pairs);
  return (int32_t)cudaGetLastError();
}

// exp_cr2 on n_pairs argument pairs (x[2i], x[2i + 1]).
extern "C" int32_t csa_selftest_exp_cr2(const float* x, float* y, int64_t n_pairs,
                                        cudaStream_t stream) {
  if (n_pairs <= 0) return 0;
  int64_t blocks = (n_pairs + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  exp_cr2_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const float2*>(x),
                                                       reinterpret_cast<float2*>(y), n_pairs);
  return (int32_t)cudaGetLastError();
}

extern "C" int32_t csa_selftest_pair_ops(const float* a, const float* b, const float* c,
                                         float* out, int64_t n_pairs, cudaStream_t stream) {
  if (n_pairs <= 0) return 0;
  int64_t blocks = (n_pairs + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  pair_ops_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      reinterpret_cast<const float2*>(a), reinterpret_cast<const float2*>(b),
      reinterpret_cast<const float2*>(c), reinterpret_cast<float2*>(out), n_pairs);
  return (int32_t)cudaGetLastError();
}

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
