/*
 * CPU oracle for the CSA/HCA fused Compressor -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library. The product path (the CUDA library under
 * gated_softmax_kv_gb300/) shares no code, header, table or helper with it.
 *
 * Subject: cuDNN-frontend "CSA Fused Compressor", sections "Semantics",
 * "Numerics" and "Support surface". The page defines
 *
 *   out[b, j] = sum_k kv[w(b,k), c(k,j)] * softmax_k(score[w(b,k), c(k,j)]
 *                                                     + ape[k % ratio, c(k,j)])
 *
 * over THD-packed segments, fp32 throughout with one final bf16 rounding.
 *
 * Two twins are provided:
 *   O32  fp32 in the plain eager order (sequential k-ascending sums from +0,
 *        every product and sum rounded separately, IEEE division, a correctly
 *        rounded exp), bf16 outputs.
 *   O64  the same loops in fp64 with no intermediate rounding, on fp64 inputs,
 *        fp64 outputs (used for finite differences and for the fp64 parity rule).
 *
 * Layouts (row-major, contiguous):
 *   kv, score   [total_tokens, coff*head_dim]   bf16 bits (uint16) / double
 *   ape         [ratio, coff*head_dim]          fp32 / double
 *   cu_seqlens, cu_seqlens_comp [num_seqs+1]    int32
 *   out         [capacity, head_dim]            bf16 bits / double
 *   grad_out    [capacity, head_dim]
 *   dkv, dscore [total_tokens, coff*head_dim]
 *   dape        [ratio, coff*head_dim]          fp32 / double
 *
 * Every entry point validates its arguments (including the caller
 * preconditions the GPU library trusts) and returns a nonzero ORACLE_E* code
 * without writing any output when they do not hold.
 */
#ifndef CSA_ORACLE_H
#define CSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  ORACLE_OK = 0,
  ORACLE_E_ARG = 1,      /* null pointer, ratio < 1, coff not in {1,2}, head_dim < 1, ... */
  ORACLE_E_SEQLENS = 2,  /* cu_seqlens not a prefix sum starting at 0 within total_tokens */
  ORACLE_E_COMP = 3,     /* cu_seqlens_comp is not the prefix sum of floor(len / ratio)   */
  ORACLE_E_CAPACITY = 4, /* capacity < true rows, or capacity > 0 with total_tokens < ratio */
};

/* Row -> window bookkeeping of one output row (exposed for the geometry pins). */
int oracle_row_map(const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                   int32_t num_seqs, int64_t row, int32_t ratio,
                   int64_t* base_token, int32_t* first_in_segment, int32_t* padding);

/* Window slot k of an output column j (exposed for the geometry pins). */
void oracle_window_slot(int32_t ratio, int32_t coff, int32_t head_dim,
                        int64_t base_token, int32_t first_in_segment,
                        int32_t j, int32_t k,
                        int64_t* token, int32_t* col, int32_t* ape_row, int32_t* valid);

/* Correctly rounded fp32 exp used by O32 (exposed for its pin). */
float oracle_exp_f32(float x);
void oracle_exp_f32_n(const float* x, float* y, int64_t n);
/* fp32 -> bf16 round-to-nearest-even, NaN -> 0x7FC0 (exposed for its pin). */
uint16_t oracle_f32_to_bf16(float x);
/* a*b + c as the oracle's translation unit evaluates it: two roundings, no FMA
 * contraction (exposed so a pin can check the build flags). */
float oracle_mul_add_f32(float a, float b, float c);

int oracle_validate(const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                    int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                    int32_t ratio, int32_t coff, int32_t head_dim);

/* O32 forward. out_f32 (nullable) receives the fp32 value before the bf16
 * rounding. nthreads <= 0 means "all cores". */
int oracle_fwd32(const uint16_t* kv, const uint16_t* score, const float* ape,
                 const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                 int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                 int32_t ratio, int32_t coff, int32_t head_dim,
                 uint16_t* out, float* out_f32, int32_t nthreads);

/* O32 backward. dape is the sum over non-padding rows of every window slot's
 * fp32 dz (masked slots included), accumulated in fp64 over fixed 64-row
 * chunks in ascending order and rounded once to fp32. */
int oracle_bwd32(const uint16_t* kv, const uint16_t* score, const float* ape,
                 const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                 int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                 int32_t ratio, int32_t coff, int32_t head_dim,
                 const uint16_t* grad_out,
                 uint16_t* dkv, uint16_t* dscore, float* dape, int32_t nthreads);

/* O64 forward / backward on fp64 inputs. */
int oracle_fwd64(const double* kv, const double* score, const double* ape,
                 const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                 int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                 int32_t ratio, int32_t coff, int32_t head_dim,
                 double* out, int32_t nthreads);

int oracle_bwd64(const double* kv, const double* score, const double* ape,
                 const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                 int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                 int32_t ratio, int32_t coff, int32_t head_dim,
                 const double* grad_out,
                 double* dkv, double* dscore, double* dape, int32_t nthreads);

#ifdef __cplusplus
}
#endif
#endif
