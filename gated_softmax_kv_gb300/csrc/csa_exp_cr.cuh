// Correctly rounded fp32 exp and division for the exact mode
// (csa_compress_fwd_exact / csa_compress_bwd_exact): with them, and with the
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
//   * N = rint(64 x / ln2), read off t = RN(x 64/ln2 + 1.5 2^23) (an
//     integer in [2^23, 2^24) for |x| <= 86, so t - 1.5 2^23 = N exactly and
//     the low bits of t's encoding hold N in two's complement: the table
//     index N mod 64 and the binary exponent k = floor(N / 64)).
//   * ln2/64 = c_hi + c2 + c3 with c_hi of 11 significant bits, so N c_hi is
//     exact (|N| < 2^13) and x - N c_hi is exact (Sterbenz); r = r_hi + r_lo
//     carries the rest in two floats (products split exactly with an FMA,
//     sums with TwoSum).
//   * e^r - 1 = r + r^2/2 + r^3 (1/6 + r/24 + r^2/120): r^2 exactly as two
//     floats, the cubic tail in fp32 (below 2^-25), as a two-float sum.
//   * 2^(j/64) = T_hi + T_lo from a 64-entry table built per CTA in fp64.
//   * y + er = T (1 + (e^r - 1)) with error below 2^-46 relative; y is the
//     correctly rounded result when y + er (1 + 2^-16) rounds to y (a
//     rounding test with a 16-fold margin on that bound), which fails for
//     about one argument in 2^17; those arguments go to fp64 exp rounded
//     once, as do NaN and |x| > 86. Arguments <= -104 (e^x < 2^-150, half
//     the smallest subnormal) give +0.
//   * The result is y 2^k (exact: y 2^k is normal for k >= -125).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_device.cuh"

namespace csa {

constexpr int kExpTableSize = 64;

// Table 2^(j/64) = hi[j] + lo[j], j = 0 .. 63, as tab[j] = hi, tab[64 + j] =
// lo in shared memory; the caller synchronises the block before the first
// exp_cr2.
__device__ __forceinline__ void exp_cr_table(float* tab) {
  const int tid = threadIdx.x + threadIdx.y * blockDim.x;
  const int nthr = blockDim.x * blockDim.y;
  for (int j = tid; j < kExpTableSize; j += nthr) {
    const double v = exp2((double)j / kExpTableSize);
    const float hi = (float)v;
    tab[j] = hi;
    tab[kExpTableSize + j] = (float)(v - (double)hi);
  }
}

// The rare path: fp64 exp rounded once, +0 far below the subnormals.
static __device__ __noinline__ float exp_cr_slow(float x) {
  return x <= -104.0f ? 0.0f : (float)exp((double)x);
}

// Correctly rounded exp of two arguments. The additions, subtractions, FMAs
// and the products that feed no addition run as two-lane instructions (each
// lane rounded as the scalar operation); the products that feed an addition
// (N c2, N c3, r r_lo, T_hi em) stay scalar, because a two-lane product may
// be fused into the two-lane addition after it (r^2 / 2 is exact, so fusing
// it changes nothing). Negated terms are formed by swapping operands (RN is
// symmetric), never by negating a register. A lane with |x| > 86 or NaN runs
// the same instructions on meaningless values (the table index stays in
// range) and takes the rare path.
__device__ __forceinline__ float2 exp_cr2(float2 x, const float* __restrict__ tab) {
  const float2 kInvC = make_float2(__int_as_float(0x42b8aa3b), __int_as_float(0x42b8aa3b));
  const float2 kShift = make_float2(12582912.0f, 12582912.0f);  // 1.5 2^23
  const float2 kMCHi = make_float2(-__int_as_float(0x3c318000), -__int_as_float(0x3c318000));
  const float kC2 = __int_as_float(0xb65e8083);
  const float2 kMC2 = make_float2(-kC2, -kC2);
  const float kC3 = __int_as_float(0x28e7bcd6);
  const float2 k6 = make_float2(__int_as_float(0x3e2aaaab), __int_as_float(0x3e2aaaab));
  const float2 k24 = make_float2(__int_as_float(0x3d2aaaab), __int_as_float(0x3d2aaaab));
  const float2 k120 = make_float2(__int_as_float(0x3c088889), __int_as_float(0x3c088889));
  const float2 kHalf = make_float2(0.5f, 0.5f), kMHalf = make_float2(-0.5f, -0.5f);
  const bool in0 = fabsf(x.x) <= 86.0f, in1 = fabsf(x.y) <= 86.0f;  // false for NaN
  // N and r = x - N ln2/64 = r_hi + r_lo
  const float2 t = fma2_rn(x, kInvC, kShift);
  const float2 nf = sub2_rn(t, kShift);  // exact
  const int b0 = __float_as_int(t.x), b1 = __float_as_int(t.y);
  const float2 rh = fma2_rn(nf, kMCHi, x);  // exact
  const float2 p = make_float2(__fmul_rn(nf.x, kC2), __fmul_rn(nf.y, kC2));
  const float2 pen = fma2_rn(nf, kMC2, p);  // p - N c2, exact: N c2 = p - pen
  const float2 s = sub2_rn(rh, p);          // TwoSum(rh, -p) = s + se
  const float2 sn = sub2_rn(p, rh);         // -s
  const float2 bb = sub2_rn(s, rh);
  const float2 se = sub2_rn(sub2_rn(rh, sub2_rn(s, bb)), add2_rn(p, bb));
  const float2 r = s;
  const float2 rl = sub2_rn(add2_rn(se, pen),
                            make_float2(__fmul_rn(nf.x, kC3), __fmul_rn(nf.y, kC3)));
  // e^r - 1 = em + eml
  const float2 r2 = mul2_rn(r, r);
  const float2 r2en = fma2_rn(sn, r, r2);  // r2 - r^2, exact: r^2 = r2 - r2en
  const float2 h = mul2_rn(kHalf, r2);     // exact
  const float2 v = fma2_rn(r, fma2_rn(r, k120, k24), k6);
  const float2 cubic = mul2_rn(mul2_rn(r2, r), v);
  const float2 em = add2_rn(r, h);  // Fast2Sum(r, h): |r| >= |h|
  const float2 emn = sub2_rn(sn, h);  // -em
  const float2 e3 = add2_rn(sub2_rn(r, em), h);
  const float2 rrl = make_float2(__fmul_rn(r.x, rl.x), __fmul_rn(r.y, rl.y));
  const float2 eml = add2_rn(add2_rn(e3, rl), add2_rn(fma2_rn(kMHalf, r2en, cubic), rrl));
  // y + er = T (1 + em + eml)
  const int i0 = b0 & (kExpTableSize - 1), i1 = b1 & (kExpTableSize - 1);
  const float2 th = make_float2(tab[i0], tab[i1]);
  const float2 tl = make_float2(tab[kExpTableSize + i0], tab[kExpTableSize + i1]);
  const float2 an = make_float2(__fmul_rn(th.x, emn.x), __fmul_rn(th.y, emn.y));  // -T_hi em
  const float2 ae = fma2_rn(th, em, an);                                          // exact
  const float2 b = add2_rn(fma2_rn(th, eml, fma2_rn(tl, em, tl)), ae);
  const float2 s2 = sub2_rn(th, an);  // Fast2Sum(T_hi, a): |T_hi| >= 1 > |a|
  const float2 e2 = sub2_rn(sub2_rn(th, s2), an);
  const float2 tt = add2_rn(e2, b);
  const float2 y = add2_rn(s2, tt);  // Fast2Sum(s2, tt)
  const float2 er = sub2_rn(tt, sub2_rn(y, s2));
  // y 2^k: k << 23 is (t's encoding << 17) with the low 23 bits cleared (the
  // index bits move there); added to y's encoding it scales y exactly, since
  // the result stays normal
  const float2 res =
      make_float2(__uint_as_float(__float_as_uint(y.x) + (((uint32_t)b0 << 17) & 0xff800000u)),
                  __uint_as_float(__float_as_uint(y.y) + (((uint32_t)b1 << 17) & 0xff800000u)));
  // rounding test (the one-sided form of CRlibm, de Dinechin, Lauter and
  // Muller): y = RN(y + er), and the exact value is within 2^-42 y of
  // y + er; if y + er (1 + 2^-16) still rounds to y, so does every value
  // within 2^-42 y of y + er (2^-42 y (1 + 2^16) stays below the distance
  // from y to the nearest midpoint for y in [0.99, 2.02])
  const float kE = __int_as_float(0x3f800080);  // 1 + 2^-16
  const float2 chk = fma2_rn(er, make_float2(kE, kE), y);
  const bool ok0 = in0 && chk.x == y.x;
  const bool ok1 = in1 && chk.y == y.y;
  if (ok0 && ok1) return res;
  return make_float2(ok0 ? res.x : exp_cr_slow(x.x), ok1 ? res.y : exp_cr_slow(x.y));
}

// p = e / den on two lanes, each correctly rounded, from y = RN(1 / den):
// div_rn_by_rcp's correction step (Markstein) where the quotient is at least
// 2^-102, IEEE division below it (the remainder would leave the fp32 range)
// and for zero, which is exact either way. den >= 1 in the softmax (the row
// maximum contributes exp(0) = 1) or NaN, which the correction carries; nden
// is -den.
__device__ __forceinline__ float2 div2_cr(float2 e, float2 den, float2 nden, float2 y) {
  const float2 q = mul2_rn(e, y);
  const float2 r = fma2_rn(nden, q, e);
  float2 p = fma2_rn(r, y, q);
  const float lo = __int_as_float(0x0c800000);  // 2^-102
  if (fminf(q.x, q.y) < lo) {
    if (q.x < lo) p.x = __fdiv_rn(e.x, den.x);
    if (q.y < lo) p.y = __fdiv_rn(e.y, den.y);
  }
  return p;
}

}  // namespace csa
