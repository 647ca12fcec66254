// Correctly rounded fp32 exp for the exact mode of the small-window kernels
// (csa_compress_fwd_exact / csa_compress_bwd_exact): with it, and with the
// eager order of operations, out, dkv and dscore are the bits of an fp32
// reference that evaluates exp in higher precision and rounds once (the
// cuDNN-frontend "CSA Fused Compressor" page aims at bit identity for ratios
// 2 and 4, section "Numerics").
//
// Method (Tang's table-driven reduction, P. T. P. Tang, "Table-driven
// implementation of the exponential function in IEEE floating-point
// arithmetic", ACM TOMS 15(2), 1989; with the rounding test of Ziv, "Fast
// evaluation of elementary mathematical functions with correctly rounded last
// bit", ACM TOMS 17(3), 1991):
//   x = (64 k + j) ln2/64 + r, |r| <= ln2/128:  exp(x) = 2^k * 2^(j/64) * e^r.
//   * N = rint(64 x / ln2); ln2/64 = c_hi + c2 + c3 with c_hi of 11
//     significant bits, so N c_hi is exact (|N| < 2^13) and x - N c_hi is
//     exact (Sterbenz); r = r_hi + r_lo carries the rest in two floats
//     (products split exactly with an FMA, sums with TwoSum).
//   * e^r - 1 = r + r^2/2 + r^3 (1/6 + r/24 + r^2/120): r^2 exactly as two
//     floats, the cubic tail in fp32 (below 2^-25), as a two-float sum.
//   * 2^(j/64) = T_hi + T_lo from a 64-entry table built per CTA in fp64.
//   * y + er = T (1 + (e^r - 1)) with error below 2^-46 relative; y is the
//     correctly rounded result unless the exact value may lie within 2^-42 of
//     a rounding boundary, which sends the argument to fp64 exp rounded once
//     (about one argument in 10^5), as do arguments outside [-86, 0] and NaN.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace csa {

constexpr int kExpTableSize = 64;

// Table 2^(j/64) = hi + lo, j = 0 .. 63, into shared memory; the caller
// synchronises the block before the first exp_cr.
__device__ __forceinline__ void exp_cr_table(float2* tab) {
  const int tid = threadIdx.x + threadIdx.y * blockDim.x;
  const int nthr = blockDim.x * blockDim.y;
  for (int j = tid; j < kExpTableSize; j += nthr) {
    const double v = exp2((double)j / kExpTableSize);
    const float hi = (float)v;
    tab[j] = make_float2(hi, (float)(v - (double)hi));
  }
}

static __device__ __noinline__ float exp_cr_slow(float x) { return (float)exp((double)x); }

__device__ __forceinline__ float exp_cr(float x, const float2* __restrict__ tab) {
  if (!(x >= -86.0f && x <= 0.0f)) return exp_cr_slow(x);  // NaN included
  const float kInvC = __int_as_float(0x42b8aa3b);  // 64 / ln2
  const float kCHi = __int_as_float(0x3c318000);   // ln2/64 to 11 bits
  const float kC2 = __int_as_float(0xb65e8083);    // next 24 bits
  const float kC3 = __int_as_float(0x28e7bcd6);    // next 24 bits
  const float k6 = __int_as_float(0x3e2aaaab);     // 1/6
  const float k24 = __int_as_float(0x3d2aaaab);    // 1/24
  const float k120 = __int_as_float(0x3c088889);   // 1/120
  const float nf = rintf(__fmul_rn(x, kInvC));
  const int n = (int)nf;
  // r = x - N ln2/64 = r_hi + r_lo
  const float rh = __fmaf_rn(-nf, kCHi, x);  // exact
  const float p = __fmul_rn(nf, kC2);
  const float pe = __fmaf_rn(nf, kC2, -p);   // N c2 = p + pe
  const float s = __fsub_rn(rh, p);           // TwoSum(rh, -p) = s + se
  const float bb = __fsub_rn(s, rh);
  const float se = __fadd_rn(__fsub_rn(rh, __fsub_rn(s, bb)), __fsub_rn(-p, bb));
  const float r = s;
  const float rl = __fsub_rn(__fsub_rn(se, pe), __fmul_rn(nf, kC3));
  // e^r - 1 = em + eml
  const float r2 = __fmul_rn(r, r);
  const float r2e = __fmaf_rn(r, r, -r2);  // r^2 = r2 + r2e
  const float h = __fmul_rn(0.5f, r2);     // exact
  const float v = __fmaf_rn(r, __fmaf_rn(r, k120, k24), k6);
  const float cubic = __fmul_rn(__fmul_rn(r2, r), v);
  const float em = __fadd_rn(r, h);  // Fast2Sum(r, h): |r| >= |h|
  const float e3 = __fadd_rn(__fsub_rn(r, em), h);
  const float eml = __fadd_rn(__fadd_rn(e3, rl),
                              __fadd_rn(__fmaf_rn(0.5f, r2e, cubic), __fmul_rn(r, rl)));
  // y + er = T (1 + em + eml)
  const float2 t = tab[n & (kExpTableSize - 1)];
  const float a = __fmul_rn(t.x, em);
  const float ae = __fmaf_rn(t.x, em, -a);
  const float b = __fadd_rn(__fmaf_rn(t.x, eml, __fmaf_rn(t.y, em, t.y)), ae);
  const float s2 = __fadd_rn(t.x, a);  // Fast2Sum(T_hi, a): |T_hi| >= 1 > |a|
  const float e2 = __fadd_rn(__fsub_rn(t.x, s2), a);
  const float tt = __fadd_rn(e2, b);
  const float y = __fadd_rn(s2, tt);  // Fast2Sum(s2, tt)
  const float er = __fsub_rn(tt, __fsub_rn(y, s2));
  // rounding test: the exact value lies within 2^-42 y of y + er; y is its
  // rounding unless that interval reaches a midpoint between y and a
  // neighbour (half an ulp away, a quarter below a power of two)
  const int yb = __float_as_int(y);
  const float half = __int_as_float((yb & 0x7f800000) - (24 << 23));
  const float room = (yb & 0x007fffff) == 0 ? __fmul_rn(0.5f, half) : half;
  if (!(__fsub_rn(room, fabsf(er)) > __fmul_rn(y, __int_as_float(0x2a800000))))  // 2^-42
    return exp_cr_slow(x);
  // 2^k with k = floor(N / 64) >= -125: exact scaling of a normal value
  return __fmul_rn(y, __int_as_float(((n >> 6) + 127) << 23));
}

}  // namespace csa
