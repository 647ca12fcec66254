// Long-window forward (window W = coff * ratio >= 16, e.g. ratio 128) of the
// CSA/HCA fused Compressor for sm_103a (cuDNN-frontend "CSA Fused
// Compressor", section "Semantics"; fp32 throughout, one final bf16 rounding).
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

namespace {

// exp of the forward kernels: the single-rounding softmax_exp_fast (the
// forward has no bitwise target).
#ifndef CSA_FWD_EXP
#define CSA_FWD_EXP softmax_exp_fast
#endif

// Long window (W >= 16): blockDim = (32, kLongRows). A lane owns 4
// consecutive columns (8-byte vectors) of a 128-column tile (blockIdx.x).
// The kLongRows warps of a CTA take kLongRows / split rows at a time, `split`
// warps per row, each warp one contiguous chunk of W / split window slots.
// A warp streams its chunk in batches of 8 slots, prefetching the next batch
// while it reduces the current one with an online softmax: running max m,
// and den and acc rescaled by exp(m_old - m_new) whenever the max grows.
// With split > 1 the chunk states (m, den, acc) meet in shared memory and the
// row's first warp merges them in chunk order (the same rescaling), so a
// problem with few output rows still has enough loads in flight; split = 1
// needs no barrier. Consecutive lanes read consecutive 8-byte columns of the
// same token row (256 bytes per warp per slot). The APE tile of the CTA (W
// slots x 128 columns) is read through L1, where it stays for the rows the
// CTA visits.
#ifndef CSA_FWD_LONG_BATCH
#define CSA_FWD_LONG_BATCH 8
#endif
#ifndef CSA_FWD_LONG_MIN_BLOCKS
#define CSA_FWD_LONG_MIN_BLOCKS 2
#endif
// kv / score loads of this kernel: the evict-first .cs form (the L1
// no-allocate form of ld_stream8 measured up to 3% slower here)
__device__ __forceinline__ uint2 long_ld8(const uint16_t* p) {
  return __ldcs(reinterpret_cast<const uint2*>(p));
}
constexpr int kLongRows = 8;                   // warps per CTA
constexpr int kBatch = CSA_FWD_LONG_BATCH;     // window slots per batch

template <int R, int COFF, int D>
__global__ void __launch_bounds__(32 * kLongRows, CSA_FWD_LONG_MIN_BLOCKS)
fwd_long_kernel(const FwdParams f, const int split) {
  grid_dependency_wait();
  allow_dependent_launch();
  constexpr int W = COFF * R;
  constexpr int NB = W / kBatch;  // batches per window, >= 2
  using S = Slot<R, COFF>;
  // chunk states by iteration parity, so one barrier per row suffices:
  // [parity][warp][m, den, acc x 4 columns][lane]
  __shared__ float part[2][kLongRows][12][32];
  const Problem& p = f.p;
  const int d = D > 0 ? D : p.d;  // D > 0: slot offsets become immediates
  const int ncv = d / 4;
  const int cv = blockIdx.x * 32 + threadIdx.x;
  const bool col_ok = cv < ncv;
  const int64_t ld = (int64_t)COFF * d;
  const int j0 = col_ok ? cv * 4 : 0;
  const float kNegInf = __int_as_float(0xff800000);
  const uint2 zero2 = make_uint2(0u, 0u);
  const uint2 ninf2 = make_uint2(kNegInfBf16x2, kNegInfBf16x2);

  const int rows_per_cta = kLongRows / split;
  const int row_local = threadIdx.y / split;
  const int chunk = threadIdx.y - row_local * split;
  const int nbc = NB / split;  // batches per chunk
  const int jb = chunk * nbc, je = jb + nbc;

  // the segment arrays in shared memory when they fit (seg_smem_bytes)
  extern __shared__ __align__(16) int32_t seg_s[];
  const SegMap sg = stage_segments(p.cu, p.cuc, p.nseq, seg_s, threadIdx.y * 32 + threadIdx.x,
                                   32 * kLongRows);
  __syncthreads();
  const int64_t true_rows = sg.cuc[p.nseq];
  const int64_t stride = (int64_t)gridDim.y * rows_per_cta;
  int hint = 0;
  int parity = 0;
  for (int64_t b0 = (int64_t)blockIdx.y * rows_per_cta; b0 < p.C; b0 += stride, parity ^= 1) {
    const int64_t b = b0 + row_local;
    const bool active = col_ok && b < p.C;
    RowInfo ri{};
    bool ok = false;
    if (active) {
      ri = row_info_from(sg.cu, sg.cuc, p.nseq, b, true_rows, R, hint);
      ok = row_in_bounds<R, COFF>(ri, p.T);
    }
    float m[4], den[4], acc[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      m[c] = kNegInf;
      den[c] = 0.0f;
      acc[c] = 0.0f;
    }
    if (ok) {
      const int64_t rowoff = ri.base * ld + j0;
      // batch j: slots [8j, 8j+8), contiguous tokens, one half of the columns
      auto load = [&](int j, uint2 (&kvb)[kBatch], uint2 (&scb)[kBatch]) {
        const int k0 = j * kBatch;
        if (S::masked(ri.first, k0)) {
#pragma unroll
          for (int t = 0; t < kBatch; ++t) {
            kvb[t] = zero2;
            scb[t] = ninf2;
          }
        } else {
          const int64_t off = rowoff + S::tok(0, k0) * ld + S::half(k0) * d;
#pragma unroll
          for (int t = 0; t < kBatch; ++t) {
            kvb[t] = long_ld8(p.kv + off + t * ld);
            scb[t] = long_ld8(p.score + off + t * ld);
          }
        }
      };
      auto reduce = [&](int j, const uint2 (&kvb)[kBatch], const uint2 (&scb)[kBatch]) {
        const int k0 = j * kBatch;
        float z[kBatch][4];
#pragma unroll
        for (int t = 0; t < kBatch; ++t) {
          const float4 a = ld_f4(p.ape + (int64_t)S::ape_row(k0 + t) * ld + S::half(k0) * d + j0);
          z[t][0] = __fadd_rn(bf16_lo(scb[t].x), a.x);
          z[t][1] = __fadd_rn(bf16_hi(scb[t].x), a.y);
          z[t][2] = __fadd_rn(bf16_lo(scb[t].y), a.z);
          z[t][3] = __fadd_rn(bf16_hi(scb[t].y), a.w);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float mn = m[c];
#pragma unroll
          for (int t = 0; t < kBatch; ++t) mn = max_nan(mn, z[t][c]);
          // while every logit so far is -inf, shift by 0 so exp gives 0, not NaN
          const float mu = mn == kNegInf ? 0.0f : mn;
          const float alpha = CSA_FWD_EXP(__fsub_rn(m[c], mu));
          float dn = __fmul_rn(den[c], alpha);
          float ac = __fmul_rn(acc[c], alpha);
#pragma unroll
          for (int t = 0; t < kBatch; ++t) {
            const float e = CSA_FWD_EXP(__fsub_rn(z[t][c], mu));
            dn = __fadd_rn(dn, e);
            ac = __fmaf_rn(e, bf16_at(c < 2 ? kvb[t].x : kvb[t].y, c & 1), ac);
          }
          m[c] = mn;
          den[c] = dn;
          acc[c] = ac;
        }
      };
      // nbc is a power of two: one batch, or an even number of them
      uint2 ka[kBatch], sa[kBatch], kb[kBatch], sb[kBatch];
      load(jb, ka, sa);
      if (nbc == 1) {
        reduce(jb, ka, sa);
      } else {
        for (int j = jb; j < je; j += 2) {
          load(j + 1, kb, sb);
          reduce(j, ka, sa);
          if (j + 2 < je) load(j + 2, ka, sa);
          reduce(j + 1, kb, sb);
        }
      }
    }
    if (split > 1) {  // uniform over the CTA
      float* mine = &part[parity][threadIdx.y][0][threadIdx.x];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        mine[c * 32] = m[c];
        mine[(4 + c) * 32] = den[c];
        mine[(8 + c) * 32] = acc[c];
      }
      __syncthreads();
      if (chunk == 0 && ok) {
        const int w0 = row_local * split;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float mx = kNegInf;
          for (int q = 0; q < split; ++q) mx = max_nan(mx, part[parity][w0 + q][c][threadIdx.x]);
          const float mu = mx == kNegInf ? 0.0f : mx;
          float dn = 0.0f, ac = 0.0f;
          for (int q = 0; q < split; ++q) {
            const float g = CSA_FWD_EXP(__fsub_rn(part[parity][w0 + q][c][threadIdx.x], mu));
            dn = __fmaf_rn(part[parity][w0 + q][4 + c][threadIdx.x], g, dn);
            ac = __fmaf_rn(part[parity][w0 + q][8 + c][threadIdx.x], g, ac);
          }
          den[c] = dn;
          acc[c] = ac;
        }
      }
    }
    if (active && chunk == 0) {
      uint16_t* dst = f.out + b * d + j0;
      if (!ok)  // violated preconditions: NaN, no access
        st_stream8(dst, make_uint2(0x7FC07FC0u, 0x7FC07FC0u));
      else
        st_stream8(dst, make_uint2(pack_bf16x2(__fdiv_rn(acc[0], den[0]), __fdiv_rn(acc[1], den[1])),
                                   pack_bf16x2(__fdiv_rn(acc[2], den[2]), __fdiv_rn(acc[3], den[3]))));
    }
  }
}

// Warps per row of the long-window forward: the smallest power of two (up to
// kLongRows and to the batches in a window) that gives at least
// CSA_FWD_SPLIT_WARPS warps over the whole problem. It depends on the problem
// only, never on the device, so results are the same on every GPU. 2048
// measured best: against 4096 it keeps one warp per row where that already
// gives 2048 warps (65536-token, head_dim 512 packs) and halves the split of
// the head_dim 128 ratio-128 packs (19.8 instead of 22.3 us at 131072 tokens,
// 21.0 instead of 22.9 us at 65536 with coff 2); 1024 loses at coff 2.
#ifndef CSA_FWD_SPLIT_WARPS
#define CSA_FWD_SPLIT_WARPS 2048
#endif

template <int R, int COFF>
cudaError_t launch_long(const FwdParams& f, cudaStream_t stream) {
  constexpr int NB = COFF * R / kBatch;
  const int ncv = f.p.d / 4;
  const int tiles = (ncv + 31) / 32;
  int split = 1;
#ifdef CSA_FWD_SPLIT_FORCE
  split = CSA_FWD_SPLIT_FORCE < NB ? CSA_FWD_SPLIT_FORCE : NB;
#else
  while (split < kLongRows && split < NB &&
         f.p.C * tiles * split < (int64_t)CSA_FWD_SPLIT_WARPS)
    split *= 2;
#endif
  auto kern = f.p.d == 512 ? fwd_long_kernel<R, COFF, 512>
             : f.p.d == 128 ? fwd_long_kernel<R, COFF, 128> : fwd_long_kernel<R, COFF, 0>;
  const int rows_per_cta = kLongRows / split;
  const size_t smem = seg_smem_bytes(f.p.nseq);
  const int occ = occupancy(reinterpret_cast<const void*>(kern), 32 * kLongRows, smem);
  const int64_t row_blocks = (f.p.C + rows_per_cta - 1) / rows_per_cta;
  int64_t gy = (int64_t)sm_count() * occ / tiles;
  if (gy < 1) gy = 1;
  if (gy > row_blocks) gy = row_blocks;
  // even out the rows per CTA: the same number of passes for every CTA
  const int64_t passes = (row_blocks + gy - 1) / gy;
  gy = (row_blocks + passes - 1) / passes;
  if (gy > 65535) gy = 65535;
  return launch_dependent(kern, dim3(tiles, (unsigned)gy), dim3(32, kLongRows), smem, stream, f, split);
}

}  // namespace

cudaError_t launch_fwd_long(const FwdParams& f, cudaStream_t stream) {
  switch (f.p.ratio * 4 + f.p.coff) {
    case 8 * 4 + 2: return launch_long<8, 2>(f, stream);
    case 16 * 4 + 1: return launch_long<16, 1>(f, stream);
    case 16 * 4 + 2: return launch_long<16, 2>(f, stream);
    case 32 * 4 + 1: return launch_long<32, 1>(f, stream);
    case 32 * 4 + 2: return launch_long<32, 2>(f, stream);
    case 64 * 4 + 1: return launch_long<64, 1>(f, stream);
    case 64 * 4 + 2: return launch_long<64, 2>(f, stream);
    case 128 * 4 + 1: return launch_long<128, 1>(f, stream);
    case 128 * 4 + 2: return launch_long<128, 2>(f, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csa
