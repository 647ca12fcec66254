// Device helpers of the bitwise kernels of the exact mode (csa_fwd_bitwise.cu,
// csa_bwd_bitwise.cu): the error bounds behind their enclosures, two-lane
// directed-rounding FMAs, the asynchronous row copies and the per-warp row
// buffer. The bounds follow from softmax_exp_fast's error envelope
// (csa_device.cuh) and the rounding error of sequential fp32 sums; each
// kernel's header states how it uses them.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_device.cuh"

namespace csa {
namespace bitwise {

constexpr int kCv = 4;  // columns per thread (8-byte words)

// softmax_exp_fast's error envelope (csa_device.cuh, checked exhaustively by
// the GPU tests): (kExpC1 |t| + kExpC0) 2^-24 relative for t in [-kTMax, 0]
constexpr float kExpC0 = kFastExpC0;
constexpr float kExpC1 = kFastExpC1;
constexpr float kTMax = kFastExpTMax;
constexpr float kU = 5.9604644775390625e-08f;  // 2^-24

template <int W>
struct Bounds {
  // p_ref / p = (1 + delta_k)(1 + Delta), with a slot's own part
  //   |delta_k| <= rho_own = (kExpC1 tau + kExpC0 + 2.5) 2^-24
  // (its exp on both sides, its product and quotient roundings) and a part
  // common to every slot of the column
  //   |Delta| <= rho_com = (kExpC0 + kExpC1 (W - 1) / e + 1.5) 2^-24
  //                        + 2^-23 (sum of den's partial sums) / den
  // (the exps' weighted contribution to den, den's roundings on both sides,
  // the reciprocal); rho = rho_own + rho_com bounds p_ref / p - 1 as a whole.
  // Every term is widened by 2^-10 (second-order terms, the inversion
  // p / p_ref -> p_ref / p and the rounding of the partial-sum ratio).
  static constexpr float kC1u = kExpC1 * kU * 1.0009765625f;
  static constexpr float kKown = (kExpC0 + 2.5f) * kU * 1.0009765625f;
  static constexpr float kKcom =
      (kExpC0 + kExpC1 * (W - 1) * 0.36787944117144233f + 1.5f) * kU * 1.0009765625f;
  static constexpr float k2u = 2.0f * kU * 1.0009765625f;
  // A slot-order sum of RN(x_k p_k) (S, or the pooled sum) then lies within
  //   sigma = ((rho_own + 2^-23) A + rho_com |sum| + 2^-23 (sum of |its partial sums|)) (1 + 2^-16)
  // of the reference's, A = sum |terms|: the common factor scales the whole
  // sum, so it counts against |sum| rather than A
  static constexpr float kWiden = 1.0000152587890625f;
};

__device__ __forceinline__ void st_u16(uint16_t* p, uint16_t v) {
  asm volatile("st.global.u16 [%0], %1;" :: "l"(p), "h"(v) : "memory");
}
// a 4-byte output store (two bf16 columns) that skips L1 allocation
__device__ __forceinline__ void st_u32_na(uint16_t* p, uint32_t v) {
  asm volatile("st.global.L1::no_allocate.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint16_t bf16_bits_rn(float x) {
  return (uint16_t)(pack_bf16x2(x, 0.0f) & 0xFFFFu);
}

// a * b + c on two lanes rounded toward -inf (RM) or +inf (RP)
#define CSA_FMA2_DIR(NAME, RND)                                                         \
  __device__ __forceinline__ float2 NAME(float2 a, float2 b, float2 c) {                \
    float2 r;                                                                           \
    asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t" \
        "mov.b64 c, {%6, %7};\n\tfma." RND ".f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}" \
        : "=f"(r.x), "=f"(r.y)                                                          \
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));                  \
    return r;                                                                           \
  }
CSA_FMA2_DIR(fma2_rm, "rm")
CSA_FMA2_DIR(fma2_rp, "rp")
#undef CSA_FMA2_DIR

// a + b, a - b, a * b on two lanes with directed rounding. Should the
// compiler fuse a product into a following sum, the fused result is the
// directed rounding of the exact value, so it stays on the same side of it.
#define CSA_OP2_DIR(NAME, OP)                                                               \
  __device__ __forceinline__ float2 NAME(float2 a, float2 b) {                              \
    float2 r;                                                                               \
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t" OP \
        " d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"                                            \
        : "=f"(r.x), "=f"(r.y)                                                              \
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                                          \
    return r;                                                                               \
  }
CSA_OP2_DIR(add2_ru, "add.rp.f32x2")
CSA_OP2_DIR(sub2_rd, "sub.rm.f32x2")
CSA_OP2_DIR(mul2_ru, "mul.rp.f32x2")
#undef CSA_OP2_DIR

__device__ __forceinline__ float2 abs2(float2 a) { return make_float2(fabsf(a.x), fabsf(a.y)); }

// A 32-bit shared-memory read the compiler cannot replace by the register
// that was stored there.
__device__ __forceinline__ uint32_t lds_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];"
               : "=r"(v) : "r"((uint32_t)__cvta_generic_to_shared(p)));
  return v;
}

// 8-byte asynchronous copies global -> shared (the next row's window, in
// flight while the current row computes), one group per row and thread
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;"
               :: "r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

// A warp's row, as copied in: the kv and score words (4 bf16 columns) of
// every slot, lane-consecutive, and grad_out; then the failing columns of the
// row as lane * 4 + column.
template <int W>
struct RowBuf {
  uint2 kv[W][32];
  uint2 sc[W][32];
  uint2 g[32];
  uint8_t fail[32 * kCv];
};

// A warp's undecided columns waiting for the exact pass, copied out of the
// row buffers so that a pass takes a full set of 64 / W columns (W / 2 lanes
// a column) whatever rows they came from: each column's window (masked slots
// as copied in: score -inf, kv 0), its output offset, its column in the
// block's APE tile and, for the backward, grad_out and the row's
// first-in-segment flag.
template <int W>
struct Pending {
  static constexpr int kCap = 64 / W;
  int64_t off[kCap];
  uint16_t sc[kCap][W];
  uint16_t kv[kCap][W];
  uint16_t tcol[kCap];
  uint16_t g[kCap];
  uint8_t first[kCap];
};

}  // namespace bitwise
}  // namespace csa
