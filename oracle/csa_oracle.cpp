/*
 * CPU oracle for the CSA/HCA fused Compressor -- TEST INFRASTRUCTURE ONLY.
 * See csa_oracle.h for the contract. Nothing under gated_softmax_kv_gb300/
 * includes, links or calls this file; only tests, the smoke check and the
 * benchmark's CPU-baseline leg do.
 *
 * Build: g++ -std=c++17 -O2 -ffp-contract=off -fno-fast-math -fopenmp
 * (no FMA contraction: every product and every sum below is rounded on its
 * own, as the page's "Numerics" section pins with mul.rn / fma.rn).
 *
 * Readings of the page that this file takes (the page is silent on them):
 *  - exp is correctly rounded in fp32: the fp64 exp rounded once to fp32;
 *  - the softmax weight is p_k = e_k / den with IEEE division;
 *  - den, the pooled sum and the backward's S are sequential k-ascending
 *    fp32 sums that start from +0;
 *  - max is NaN-propagating;
 *  - a masked window slot (previous block of a segment's first block,
 *    coff == 2) enters as kv = 0 and score = -inf, so its logit is
 *    -inf + ape and its dz (= p * (dp - S) = 0 * (0 - S)) still enters dape;
 *  - a padding row (row >= cu_seqlens_comp[-1]) is "first in segment from
 *    token 0": base token 0, previous-block slots masked.
 */
#include "csa_oracle.h"

#include <cfloat>
#include <cmath>
#include <cstring>
#include <limits>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the fp32 oracle needs float expressions evaluated in float"
#endif

namespace {

const int64_t kDapeChunkRows = 64;  // fixed row chunk of the dape sum

float bf16_bits_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

float nan_max_f(float a, float b) {
  if (std::isnan(a) || std::isnan(b)) return std::numeric_limits<float>::quiet_NaN();
  return a < b ? b : a;
}

double nan_max_d(double a, double b) {
  if (std::isnan(a) || std::isnan(b)) return std::numeric_limits<double>::quiet_NaN();
  return a < b ? b : a;
}

int pick_threads(int32_t nthreads) {
#ifdef _OPENMP
  return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/* One window slot, resolved: where it reads and whether it is masked. */
struct Slot {
  int64_t token;
  int32_t col;
  int32_t ape_row;
  int32_t valid;
};

void resolve_window(int32_t ratio, int32_t coff, int32_t head_dim, int64_t base,
                    int32_t first, int32_t j, std::vector<Slot>& slots) {
  const int32_t width = coff * ratio;
  slots.resize(width);
  for (int32_t k = 0; k < width; ++k) {
    Slot& s = slots[k];
    oracle_window_slot(ratio, coff, head_dim, base, first, j, k, &s.token, &s.col,
                       &s.ape_row, &s.valid);
  }
}

/* Rows that carry a gradient: non-padding rows that have an output slot. */
int64_t grad_rows(const int32_t* cuc, int32_t num_seqs, int64_t capacity) {
  int64_t true_rows = cuc[num_seqs];
  return true_rows < capacity ? true_rows : capacity;
}

}  // namespace

extern "C" {

float oracle_exp_f32(float x) { return (float)std::exp((double)x); }

void oracle_exp_f32_n(const float* x, float* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_exp_f32(x[i]);
}

uint16_t oracle_f32_to_bf16(float x) {
  if (std::isnan(x)) return 0x7FC0;
  uint32_t u;
  std::memcpy(&u, &x, sizeof u);
  uint32_t upper = u >> 16;
  uint32_t lower = u & 0xFFFFu;
  // round half to even on the 16 dropped bits; a carry into the exponent is
  // the correct next binade (and turns the largest finite values into inf)
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

/* a*b + c as this translation unit evaluates it (a pin checks: two roundings). */
float oracle_mul_add_f32(float a, float b, float c) { return a * b + c; }

int oracle_row_map(const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                   int32_t num_seqs, int64_t row, int32_t ratio, int64_t* base_token,
                   int32_t* first_in_segment, int32_t* padding) {
  const int64_t true_rows = cu_seqlens_comp[num_seqs];
  if (row < true_rows) {
    for (int32_t s = 0; s < num_seqs; ++s) {
      if (cu_seqlens_comp[s] <= row && row < cu_seqlens_comp[s + 1]) {
        const int64_t i = row - cu_seqlens_comp[s];  // block index inside segment s
        *base_token = (int64_t)cu_seqlens[s] + i * ratio;
        *first_in_segment = (i == 0);
        *padding = 0;
        return ORACLE_OK;
      }
    }
    return ORACLE_E_COMP;
  }
  // static-capacity padding row: first-in-segment semantics from token 0
  *base_token = 0;
  *first_in_segment = 1;
  *padding = 1;
  return ORACLE_OK;
}

void oracle_window_slot(int32_t ratio, int32_t coff, int32_t head_dim, int64_t base_token,
                        int32_t first_in_segment, int32_t j, int32_t k, int64_t* token,
                        int32_t* col, int32_t* ape_row, int32_t* valid) {
  if (coff == 2 && k < ratio) {
    // previous block's token, first-half column, APE row k; masked on a first block
    *token = base_token - ratio + k;
    *col = j;
    *ape_row = k;
    *valid = !first_in_segment;
  } else if (coff == 2) {
    // own block's token, second-half column, APE row k - ratio
    *token = base_token + (k - ratio);
    *col = head_dim + j;
    *ape_row = k - ratio;
    *valid = 1;
  } else {
    // own-block window: own token, column j, APE row k, always valid
    *token = base_token + k;
    *col = j;
    *ape_row = k;
    *valid = 1;
  }
}

int oracle_validate(const int32_t* cu, const int32_t* cuc, int32_t num_seqs,
                    int64_t total_tokens, int64_t capacity, int32_t ratio, int32_t coff,
                    int32_t head_dim) {
  if (!cu || !cuc) return ORACLE_E_ARG;
  if (num_seqs < 1 || ratio < 1 || (coff != 1 && coff != 2) || head_dim < 1) return ORACLE_E_ARG;
  if (total_tokens < 0 || capacity < 0) return ORACLE_E_ARG;
  if (cu[0] != 0) return ORACLE_E_SEQLENS;
  for (int32_t s = 0; s < num_seqs; ++s)
    if (cu[s + 1] < cu[s]) return ORACLE_E_SEQLENS;
  if (cu[num_seqs] > total_tokens) return ORACLE_E_SEQLENS;
  if (cuc[0] != 0) return ORACLE_E_COMP;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int64_t len = (int64_t)cu[s + 1] - cu[s];
    if ((int64_t)cuc[s + 1] - cuc[s] != len / ratio) return ORACLE_E_COMP;
  }
  if ((int64_t)cuc[num_seqs] > capacity) return ORACLE_E_CAPACITY;
  if (capacity > 0 && total_tokens < ratio) return ORACLE_E_CAPACITY;
  return ORACLE_OK;
}

/* ---------------------------------------------------------------- O32 --- */

int oracle_fwd32(const uint16_t* kv, const uint16_t* score, const float* ape,
                 const int32_t* cu, const int32_t* cuc, int32_t num_seqs,
                 int64_t total_tokens, int64_t capacity, int32_t ratio, int32_t coff,
                 int32_t head_dim, uint16_t* out, float* out_f32, int32_t nthreads) {
  if (!kv || !score || !ape || !out) return ORACLE_E_ARG;
  int rc = oracle_validate(cu, cuc, num_seqs, total_tokens, capacity, ratio, coff, head_dim);
  if (rc != ORACLE_OK) return rc;
  const int64_t ld = (int64_t)coff * head_dim;  // packed row width of kv / score / ape
  const int32_t width = coff * ratio;

#pragma omp parallel num_threads(pick_threads(nthreads))
  {
    std::vector<Slot> slots;
    std::vector<float> x(width), z(width), e(width), p(width);
#pragma omp for schedule(static)
    for (int64_t b = 0; b < capacity; ++b) {
      int64_t base;
      int32_t first, pad;
      oracle_row_map(cu, cuc, num_seqs, b, ratio, &base, &first, &pad);
      for (int32_t j = 0; j < head_dim; ++j) {
        resolve_window(ratio, coff, head_dim, base, first, j, slots);
        for (int32_t k = 0; k < width; ++k) {
          const Slot& s = slots[k];
          const float xk = s.valid ? bf16_bits_to_f32(kv[s.token * ld + s.col]) : 0.0f;
          const float sk = s.valid ? bf16_bits_to_f32(score[s.token * ld + s.col])
                                   : -std::numeric_limits<float>::infinity();
          x[k] = xk;
          z[k] = sk + ape[(int64_t)s.ape_row * ld + s.col];
        }
        float m = z[0];
        for (int32_t k = 1; k < width; ++k) m = nan_max_f(m, z[k]);
        for (int32_t k = 0; k < width; ++k) e[k] = oracle_exp_f32(z[k] - m);
        float den = 0.0f;
        for (int32_t k = 0; k < width; ++k) den = den + e[k];
        for (int32_t k = 0; k < width; ++k) p[k] = e[k] / den;
        float acc = 0.0f;
        for (int32_t k = 0; k < width; ++k) {
          const float term = p[k] * x[k];
          acc = acc + term;
        }
        out[b * head_dim + j] = oracle_f32_to_bf16(acc);
        if (out_f32) out_f32[b * head_dim + j] = acc;
      }
    }
  }
  return ORACLE_OK;
}

int oracle_bwd32(const uint16_t* kv, const uint16_t* score, const float* ape,
                 const int32_t* cu, const int32_t* cuc, int32_t num_seqs,
                 int64_t total_tokens, int64_t capacity, int32_t ratio, int32_t coff,
                 int32_t head_dim, const uint16_t* grad_out, uint16_t* dkv, uint16_t* dscore,
                 float* dape, int32_t nthreads) {
  if (!kv || !score || !ape || !grad_out || !dkv || !dscore || !dape) return ORACLE_E_ARG;
  int rc = oracle_validate(cu, cuc, num_seqs, total_tokens, capacity, ratio, coff, head_dim);
  if (rc != ORACLE_OK) return rc;
  const int64_t ld = (int64_t)coff * head_dim;
  const int32_t width = coff * ratio;
  const int64_t n_ape = (int64_t)ratio * ld;

  // every position no row writes is an exact +0
  std::memset(dkv, 0, sizeof(uint16_t) * total_tokens * ld);
  std::memset(dscore, 0, sizeof(uint16_t) * total_tokens * ld);

  const int64_t rows = grad_rows(cuc, num_seqs, capacity);  // padding rows carry no gradient
  const int64_t n_chunks = (rows + kDapeChunkRows - 1) / kDapeChunkRows;
  std::vector<double> partial((size_t)(n_chunks > 0 ? n_chunks : 1) * n_ape, 0.0);

#pragma omp parallel num_threads(pick_threads(nthreads))
  {
    std::vector<Slot> slots;
    std::vector<float> x(width), z(width), e(width), p(width), dp(width);
#pragma omp for schedule(static)
    for (int64_t c = 0; c < n_chunks; ++c) {
      double* part = &partial[(size_t)c * n_ape];
      const int64_t b_end = (c + 1) * kDapeChunkRows < rows ? (c + 1) * kDapeChunkRows : rows;
      for (int64_t b = c * kDapeChunkRows; b < b_end; ++b) {
        int64_t base;
        int32_t first, pad;
        oracle_row_map(cu, cuc, num_seqs, b, ratio, &base, &first, &pad);
        for (int32_t j = 0; j < head_dim; ++j) {
          resolve_window(ratio, coff, head_dim, base, first, j, slots);
          // forward recompute, same order as oracle_fwd32
          for (int32_t k = 0; k < width; ++k) {
            const Slot& s = slots[k];
            const float xk = s.valid ? bf16_bits_to_f32(kv[s.token * ld + s.col]) : 0.0f;
            const float sk = s.valid ? bf16_bits_to_f32(score[s.token * ld + s.col])
                                     : -std::numeric_limits<float>::infinity();
            x[k] = xk;
            z[k] = sk + ape[(int64_t)s.ape_row * ld + s.col];
          }
          float m = z[0];
          for (int32_t k = 1; k < width; ++k) m = nan_max_f(m, z[k]);
          for (int32_t k = 0; k < width; ++k) e[k] = oracle_exp_f32(z[k] - m);
          float den = 0.0f;
          for (int32_t k = 0; k < width; ++k) den = den + e[k];
          for (int32_t k = 0; k < width; ++k) p[k] = e[k] / den;
          // softmax-pool backward
          const float g = bf16_bits_to_f32(grad_out[b * head_dim + j]);
          float S = 0.0f;
          for (int32_t k = 0; k < width; ++k) {
            dp[k] = g * x[k];
            const float term = dp[k] * p[k];
            S = S + term;
          }
          for (int32_t k = 0; k < width; ++k) {
            const Slot& s = slots[k];
            const float diff = dp[k] - S;
            const float dz = p[k] * diff;
            const float dkvk = g * p[k];
            if (s.valid) {
              dkv[s.token * ld + s.col] = oracle_f32_to_bf16(dkvk);
              dscore[s.token * ld + s.col] = oracle_f32_to_bf16(dz);
            }
            part[(int64_t)s.ape_row * ld + s.col] += (double)dz;
          }
        }
      }
    }
  }
  for (int64_t i = 0; i < n_ape; ++i) {
    double sum = 0.0;
    for (int64_t c = 0; c < n_chunks; ++c) sum += partial[(size_t)c * n_ape + i];
    dape[i] = (float)sum;
  }
  return ORACLE_OK;
}

/* ---------------------------------------------------------------- O64 --- */

int oracle_fwd64(const double* kv, const double* score, const double* ape,
                 const int32_t* cu, const int32_t* cuc, int32_t num_seqs,
                 int64_t total_tokens, int64_t capacity, int32_t ratio, int32_t coff,
                 int32_t head_dim, double* out, int32_t nthreads) {
  if (!kv || !score || !ape || !out) return ORACLE_E_ARG;
  int rc = oracle_validate(cu, cuc, num_seqs, total_tokens, capacity, ratio, coff, head_dim);
  if (rc != ORACLE_OK) return rc;
  const int64_t ld = (int64_t)coff * head_dim;
  const int32_t width = coff * ratio;

#pragma omp parallel num_threads(pick_threads(nthreads))
  {
    std::vector<Slot> slots;
    std::vector<double> x(width), z(width), e(width);
#pragma omp for schedule(static)
    for (int64_t b = 0; b < capacity; ++b) {
      int64_t base;
      int32_t first, pad;
      oracle_row_map(cu, cuc, num_seqs, b, ratio, &base, &first, &pad);
      for (int32_t j = 0; j < head_dim; ++j) {
        resolve_window(ratio, coff, head_dim, base, first, j, slots);
        for (int32_t k = 0; k < width; ++k) {
          const Slot& s = slots[k];
          x[k] = s.valid ? kv[s.token * ld + s.col] : 0.0;
          const double sk = s.valid ? score[s.token * ld + s.col]
                                    : -std::numeric_limits<double>::infinity();
          z[k] = sk + ape[(int64_t)s.ape_row * ld + s.col];
        }
        double m = z[0];
        for (int32_t k = 1; k < width; ++k) m = nan_max_d(m, z[k]);
        double den = 0.0;
        for (int32_t k = 0; k < width; ++k) {
          e[k] = std::exp(z[k] - m);
          den += e[k];
        }
        double acc = 0.0;
        for (int32_t k = 0; k < width; ++k) acc += (e[k] / den) * x[k];
        out[b * head_dim + j] = acc;
      }
    }
  }
  return ORACLE_OK;
}

int oracle_bwd64(const double* kv, const double* score, const double* ape,
                 const int32_t* cu, const int32_t* cuc, int32_t num_seqs,
                 int64_t total_tokens, int64_t capacity, int32_t ratio, int32_t coff,
                 int32_t head_dim, const double* grad_out, double* dkv, double* dscore,
                 double* dape, int32_t nthreads) {
  if (!kv || !score || !ape || !grad_out || !dkv || !dscore || !dape) return ORACLE_E_ARG;
  int rc = oracle_validate(cu, cuc, num_seqs, total_tokens, capacity, ratio, coff, head_dim);
  if (rc != ORACLE_OK) return rc;
  const int64_t ld = (int64_t)coff * head_dim;
  const int32_t width = coff * ratio;
  const int64_t n_ape = (int64_t)ratio * ld;

  for (int64_t i = 0; i < total_tokens * ld; ++i) {
    dkv[i] = 0.0;
    dscore[i] = 0.0;
  }
  const int64_t rows = grad_rows(cuc, num_seqs, capacity);
  const int64_t n_chunks = (rows + kDapeChunkRows - 1) / kDapeChunkRows;
  std::vector<double> partial((size_t)(n_chunks > 0 ? n_chunks : 1) * n_ape, 0.0);

#pragma omp parallel num_threads(pick_threads(nthreads))
  {
    std::vector<Slot> slots;
    std::vector<double> x(width), z(width), p(width), dp(width);
#pragma omp for schedule(static)
    for (int64_t c = 0; c < n_chunks; ++c) {
      double* part = &partial[(size_t)c * n_ape];
      const int64_t b_end = (c + 1) * kDapeChunkRows < rows ? (c + 1) * kDapeChunkRows : rows;
      for (int64_t b = c * kDapeChunkRows; b < b_end; ++b) {
        int64_t base;
        int32_t first, pad;
        oracle_row_map(cu, cuc, num_seqs, b, ratio, &base, &first, &pad);
        for (int32_t j = 0; j < head_dim; ++j) {
          resolve_window(ratio, coff, head_dim, base, first, j, slots);
          for (int32_t k = 0; k < width; ++k) {
            const Slot& s = slots[k];
            x[k] = s.valid ? kv[s.token * ld + s.col] : 0.0;
            const double sk = s.valid ? score[s.token * ld + s.col]
                                      : -std::numeric_limits<double>::infinity();
            z[k] = sk + ape[(int64_t)s.ape_row * ld + s.col];
          }
          double m = z[0];
          for (int32_t k = 1; k < width; ++k) m = nan_max_d(m, z[k]);
          double den = 0.0;
          for (int32_t k = 0; k < width; ++k) {
            p[k] = std::exp(z[k] - m);
            den += p[k];
          }
          for (int32_t k = 0; k < width; ++k) p[k] = p[k] / den;
          const double g = grad_out[b * head_dim + j];
          double S = 0.0;
          for (int32_t k = 0; k < width; ++k) {
            dp[k] = g * x[k];
            S += dp[k] * p[k];
          }
          for (int32_t k = 0; k < width; ++k) {
            const Slot& s = slots[k];
            const double dz = p[k] * (dp[k] - S);
            if (s.valid) {
              dkv[s.token * ld + s.col] = g * p[k];
              dscore[s.token * ld + s.col] = dz;
            }
            part[(int64_t)s.ape_row * ld + s.col] += dz;
          }
        }
      }
    }
  }
  for (int64_t i = 0; i < n_ape; ++i) {
    double sum = 0.0;
    for (int64_t c = 0; c < n_chunks; ++c) sum += partial[(size_t)c * n_ape + i];
    dape[i] = sum;
  }
  return ORACLE_OK;
}

}  // extern "C"
