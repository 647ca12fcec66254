// Device-side building blocks shared by the forward and backward kernels of
// the CSA/HCA fused Compressor (cuDNN-frontend "CSA Fused Compressor").
//
// Numerics (page section "Numerics"): every product, sum and quotient is a
// separately rounded fp32 operation (__fmul_rn / __fadd_rn / __fsub_rn /
// __fdiv_rn, so no FMA contraction can change a result), max propagates NaN,
// bf16 values widen exactly and narrow once with round-to-nearest-even.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_internal.h"

namespace csa {

constexpr int kVec = 8;                  // bf16 elements per 16-byte vector
constexpr uint32_t kNegInfBf16x2 = 0xFF80FF80u;

// ---- bf16 <-> fp32 ---------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_at(uint32_t w, int h) { return h ? bf16_hi(w) : bf16_lo(w); }


// Two fp32 values -> one bf16x2 word (lo at the lower address), nearest-even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// ---- exp --------------------------------------------------------------------

__device__ __forceinline__ float ex2_approx_ftz(float t) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
  return r;
}

// exp(x) for the softmax weights, x = z - max <= 0 (or NaN).
// exp(x) = 2^(x * log2 e). The product x * log2 e is carried beyond fp32
// precision as t + err: log2 e is split into an fp32 head and tail, and the
// head product's rounding error is recovered exactly with one FMA (the
// TwoProduct step of Ogita, Rump & Oishi, "Accurate sum and dot product",
// SIAM J. Sci. Comput. 26(6), 2005). Then 2^(t + err) = 2^t * (1 + err ln 2)
// to first order (|err| <= 2^-17 here, so the dropped term is below 2^-35),
// with 2^t from the hardware ex2.approx. x is clamped at -100 (exp(-100) is
// below the smallest fp32 subnormal; ftz flushes results below 2^-126 to 0)
// with a NaN-propagating max, so -inf gives 0 and NaN stays NaN.
__device__ __forceinline__ float softmax_exp(float x) {
  const float kLog2eHi = __int_as_float(0x3fb8aa3b);  // fp32(log2 e)
  const float kLog2eLo = __int_as_float(0x32a57060);  // log2 e - kLog2eHi
  const float kLn2 = __int_as_float(0x3f317218);      // fp32(ln 2)
  x = max_nan(x, -100.0f);
  const float t = __fmul_rn(x, kLog2eHi);
  float err = __fmaf_rn(x, kLog2eHi, -t);
  err = __fmaf_rn(x, kLog2eLo, err);
  const float r = ex2_approx_ftz(t);
  return __fmaf_rn(r, __fmul_rn(err, kLn2), r);
}

// exp(x) as 2^(x log2 e) with a single rounding of the product (no error
// term): relative error about |x| 2^-24 from the product plus that of
// ex2.approx. No clamp: ex2.approx.ftz gives +0 for -inf and flushes every
// result below 2^-126 (all x < -87.4) to +0, and NaN stays NaN.
__device__ __forceinline__ float softmax_exp_fast(float x) {
  return ex2_approx_ftz(__fmul_rn(x, __int_as_float(0x3fb8aa3b)));
}

// Error envelope of softmax_exp_fast used by the bitwise backward: for every
// fp32 x in [-kFastExpTMax, 0], |softmax_exp_fast(x) / CR(exp(x)) - 1| <=
// (kFastExpC1 |x| + kFastExpC0) 2^-24, CR the correctly rounded result. The
// |x| term is fp32(log2 e)'s error (0.22 ulp) plus the rounding of x log2 e
// (together at most 1.23 |x| ulp of the result); the constant covers
// ex2.approx's own error and the correct rounding. The GPU tests check the
// envelope on every fp32 x of the range.
constexpr float kFastExpC0 = 3.25f;
constexpr float kFastExpC1 = 1.25f;
constexpr float kFastExpTMax = 60.0f;

// ---- paired fp32 arithmetic --------------------------------------------------

// Two independent fp32 operations in one instruction (the f32x2 forms of the
// sm_100 family). Each lane is rounded to nearest exactly as __fadd_rn /
// __fsub_rn / __fmul_rn / __fmaf_rn would round it. Unlike the scalar _rn
// forms, a two-lane product followed by a two-lane add or subtract may be
// fused into one FMA by the compiler (measured), so callers never chain them
// that way; every other use gives the scalar bits with half the instructions.
#define CSA_F32X2_OP(NAME, OP)                                                              \
  __device__ __forceinline__ float2 NAME(float2 a, float2 b) {                              \
    float2 r;                                                                               \
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t" OP \
        " d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"                                            \
        : "=f"(r.x), "=f"(r.y)                                                              \
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                                          \
    return r;                                                                               \
  }
CSA_F32X2_OP(add2_rn, "add.rn.f32x2")
CSA_F32X2_OP(sub2_rn, "sub.rn.f32x2")
CSA_F32X2_OP(mul2_rn, "mul.rn.f32x2")
#undef CSA_F32X2_OP

__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mov.b64 c, {%6, %7};\n\tfma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

// softmax_exp_fast on two lanes: the products x * log2 e in one instruction.
__device__ __forceinline__ float2 softmax_exp_fast2(float2 x) {
  const float l = __int_as_float(0x3fb8aa3b);
  const float2 t = mul2_rn(x, make_float2(l, l));
  return make_float2(ex2_approx_ftz(t.x), ex2_approx_ftz(t.y));
}

// ---- bf16 inputs, three-input max / min ------------------------------------

// The two bf16 halves of a word (lower address first) as 16-bit registers.
__device__ __forceinline__ void split_bf16x2(uint32_t w, uint16_t& lo, uint16_t& hi) {
  asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(w));
}
__device__ __forceinline__ uint16_t bf16_half(uint32_t w, int h) {
  uint16_t lo, hi;
  split_bf16x2(w, lo, hi);
  return h ? hi : lo;
}
// Mixed-precision forms of the sm_100 family, bf16 inputs read as fp32:
// RN(a + c) and RN(a b + c). A product of two bf16 values is exact in fp32,
// so with c = -0 the FMA gives RN(a b), signed zeros included.
__device__ __forceinline__ float add_bf16_f32(uint16_t a, float c) {
  float d;
  asm("add.rn.f32.bf16 %0, %1, %2;" : "=f"(d) : "h"(a), "f"(c));
  return d;
}
__device__ __forceinline__ float mul_bf16(uint16_t a, uint16_t b) {
  float d;
  asm("fma.rn.f32.bf16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(-0.0f));
  return d;
}
// Three-input max propagating NaN (as max_nan) and min skipping it (as fminf).
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Max / min of v[lo, hi) (hi - lo >= 1) with the three-input forms.
template <int LO, int HI, class F>
__device__ __forceinline__ float max_range(F v) {
  float m = v(LO);
#pragma unroll
  for (int k = LO + 1; k < HI; k += 2) m = (k + 1 < HI) ? max3_nan(m, v(k), v(k + 1)) : max_nan(m, v(k));
  return m;
}
template <int LO, int HI, class F>
__device__ __forceinline__ float min_range(F v) {
  float m = v(LO);
#pragma unroll
  for (int k = LO + 1; k < HI; k += 2) m = (k + 1 < HI) ? min3(m, v(k), v(k + 1)) : fminf(m, v(k));
  return m;
}

// ---- division ---------------------------------------------------------------

// a / b rounded to nearest from y = RN(1/b): q = RN(a*y), then one
// correction step with the exact remainder r = a - b*q (an FMA computes it
// exactly), q' = RN(q + r*y). With y the correctly rounded reciprocal this
// returns the correctly rounded quotient when nothing overflows or
// underflows (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990; the theorem is
// restated in Muller et al., "Handbook of Floating-Point Arithmetic",
// section on Newton-Raphson-based division with an FMA). The theorem needs
// the remainder to be exact: its last bit is ulp(b) * ulp(q), which stays in
// fp32 range when the quotient is at least 2^-103 (b >= 1). Below that the
// result can be one ulp off. The softmax uses it with a = e in [0, 1] and
// b = den in [1, W], where one reciprocal per column serves all W slots; a
// weight below 2^-103 is the only case outside the correctly rounded domain.
__device__ __forceinline__ float div_rn_by_rcp(float a, float b, float y) {
  const float q = __fmul_rn(a, y);
  const float r = __fmaf_rn(-b, q, a);
  return __fmaf_rn(r, y, q);
}

// ---- programmatic dependent launch -------------------------------------------

// Every kernel of the library is launched with programmatic stream
// serialization (launch_dependent below): it may become resident while the
// previous kernel on the stream drains, and grid_dependency_wait holds it
// until that grid has completed and its memory operations are visible. So
// each kernel calls it before its first global access (read or write), and
// allow_dependent_launch right after, letting the next kernel's launch
// overlap this one's tail (it can only start once every CTA of this grid
// has started). Both are no-ops under a normal launch.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- memory ----------------------------------------------------------------

// kv / score / grad_out are read exactly once: streaming (evict-first) loads.
// Streaming loads of kv / score / grad_out: read once, so they take no L1
// line (L1::no_allocate; measured 1.1% faster forward and 0.6% faster
// backward at the 256k-token headline than the evict-first .cs form).
__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) {
  uint4 v;
  asm("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
// Streaming stores of out / dkv / dscore: no L1 line and the normal L2 policy
// (measured 1.0% faster backward at the headline than the evict-first .cs
// form, which the plain form was not).
__device__ __forceinline__ void st_stream(uint16_t* p, uint4 v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ uint2 ld_stream8(const uint16_t* p) {
  uint2 v;
  asm("ld.global.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream8(uint16_t* p, uint2 v) {
  asm volatile("st.global.L1::no_allocate.v2.u32 [%0], {%1, %2};" :: "l"(p), "r"(v.x), "r"(v.y)
               : "memory");
}
__device__ __forceinline__ float4 ld_f4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

// ---- row -> segment map (page section "Semantics") -------------------------

struct RowInfo {
  int64_t base;      // first token of the row's own block
  int64_t seg_end;   // cu_seqlens[s + 1] (0 for padding rows)
  bool first;        // first block of its segment (or a padding row)
  bool last;         // last block of its segment
};

// The segment arrays as a kernel reads them: a CTA's copy in shared memory
// when each has at most kSegSmemMax entries, else the caller's global arrays.
// A row's lookup (below) then costs shared-memory reads instead of dependent
// L2 or DRAM loads ahead of the row's own loads; the copy is one round trip in
// the prologue, next to the APE slice.
constexpr int kSegSmemMax = 1024;
__host__ __device__ inline size_t seg_smem_stride(int nseq) {  // entries, 16-byte multiple
  return ((size_t)(nseq + 1) + 3) / 4 * 4;
}
__host__ __device__ inline size_t seg_smem_bytes(int nseq) {
  return nseq + 1 <= kSegSmemMax ? 2 * sizeof(int32_t) * seg_smem_stride(nseq) : 0;
}
constexpr size_t kSegSmemBytesMax = 2 * sizeof(int32_t) * kSegSmemMax;  // seg_smem_bytes' bound
struct SegMap {
  const int32_t* cu;   // cu_seqlens[0 .. nseq]
  const int32_t* cuc;  // cu_seqlens_comp[0 .. nseq]
};
// Copies the arrays into s (seg_smem_bytes(nseq) bytes, 16-byte aligned) when
// they fit; the copy is readable after the caller's next __syncthreads.
__device__ __forceinline__ SegMap stage_segments(const int32_t* cu, const int32_t* cuc, int nseq,
                                                 int32_t* s, int tid, int nthr) {
  const int n = nseq + 1;
  if (n > kSegSmemMax) return SegMap{cu, cuc};
  const int stride = (int)seg_smem_stride(nseq);
  for (int i = tid; i < n; i += nthr) {
    s[i] = __ldg(cu + i);
    s[stride + i] = __ldg(cuc + i);
  }
  return SegMap{s, s + stride};
}

// Row b < true_rows: s = last segment with cu_seqlens_comp[s] <= b,
// i = b - cu_seqlens_comp[s], base = cu_seqlens[s] + i * ratio.
// Row b >= true_rows (static-capacity padding): first block from token 0.
// For a thread that visits rows in increasing order: `hint` is a segment with
// cu_seqlens_comp[hint] <= b from an earlier row (0 at first); the common case
// costs one load, otherwise a binary search over the later segments, which
// terminates and stays in [0, num_seqs) whatever the arrays hold. cu and cuc
// are generic pointers (a SegMap's shared-memory copy or the global arrays);
// with kGlobalRO they must be the global arrays, read through the read-only
// path (loads the compiler may hoist past the kernel's own stores).
template <bool kGlobalRO = false>
__device__ __forceinline__ RowInfo row_info_from(const int32_t* cu, const int32_t* cuc, int nseq,
                                                 int64_t b, int64_t true_rows, int ratio,
                                                 int& hint) {
  auto ld = [](const int32_t* q) -> int32_t { return kGlobalRO ? __ldg(q) : *q; };
  RowInfo ri;
  if (b >= true_rows) {
    ri.base = 0;
    ri.seg_end = 0;
    ri.first = true;
    ri.last = false;
    return ri;
  }
  int lo = hint;
  int64_t c1 = ld(cuc + lo + 1);
  if (c1 <= b) {
    int hi = nseq;
    lo = lo + 1;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if ((int64_t)ld(cuc + mid) <= b) lo = mid; else hi = mid;
    }
    c1 = ld(cuc + lo + 1);
  }
  hint = lo;
  const int64_t c0 = ld(cuc + lo);
  const int64_t i = b - c0;
  ri.base = (int64_t)ld(cu + lo) + i * ratio;
  ri.seg_end = ld(cu + lo + 1);
  ri.first = (i == 0);
  ri.last = (i == c1 - c0 - 1);
  return ri;
}

// Window slot k of a row: token offset from base, column offset (0 or d),
// APE row; masked when it is a previous-block slot of a first block.
template <int R, int COFF>
struct Slot {
  static __device__ __forceinline__ int64_t tok(int64_t base, int k) {
    return COFF == 2 ? (k < R ? base - R + k : base + (k - R)) : base + k;
  }
  static __device__ __forceinline__ int half(int k) { return (COFF == 2 && k >= R) ? 1 : 0; }
  static __device__ __forceinline__ int ape_row(int k) { return (COFF == 2 && k >= R) ? k - R : k; }
  static __device__ __forceinline__ bool masked(bool first, int k) {
    return COFF == 2 && k < R && first;
  }
};

// Every token a row touches must lie in [0, T): false means violated caller
// preconditions; such a row is skipped rather than read out of bounds.
template <int R, int COFF>
__device__ __forceinline__ bool row_in_bounds(const RowInfo& ri, int64_t T) {
  const int64_t lo = (COFF == 2 && !ri.first) ? ri.base - R : ri.base;
  return lo >= 0 && ri.base + R <= T;
}

}  // namespace csa
