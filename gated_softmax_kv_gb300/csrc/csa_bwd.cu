// Backward kernels of the CSA/HCA fused Compressor for sm_103a.
//
// cuDNN-frontend "CSA Fused Compressor", sections "Semantics" and "Class API":
// with p the softmax weights of a row's window, g = grad_out[b, j],
//   dp_k = g * kv_k,  S = sum_k dp_k * p_k,
//   dscore_k = p_k * (dp_k - S),  dkv_k = g * p_k,  dape[k % ratio, c] += dscore_k.
// dkv / dscore are written in full: every position a non-padding row reads
// gets its gradient from that row (the unique reader), every other position
// gets +0 from a unique owner -- the segment's last row owns its block's
// unread first-half columns and the segment tail, and a sweep over segments
// shorter than `ratio` and over tokens >= cu_seqlens[-1] owns the rest.
// Padding rows (b >= cu_seqlens_comp[-1]) are not visited at all.
//
// dape is reduced deterministically in two levels, without atomics: each CTA
// accumulates its rows' logit gradients (rows in a fixed order; registers in
// bwd_small, a shared-memory table in bwd_long), combines its threads in a
// fixed order and writes one fp32 partial per row group; dape_reduce then
// sums the partials in a fixed order and overwrites dape.
//
// Kernel shapes mirror the forward (csa_fwd.cu): bwd_small keeps a W <= 8
// window of 4 columns per thread in registers and follows the eager
// operation order (m, e, den, p = e * (1 / den), sequential sums); bwd_long
// splits W >= 16 windows over warps of 8 or 16 slots, merges the per-chunk
// (max, sum exp, sum (g kv) exp) triples in a fixed order through shared
// memory and prefetches the next row while it computes the current one.
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_bwd_common.cuh"
#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

namespace {

constexpr int kThreads = 256;

// exp and division of the small-window backward's per-element weights. The
// default is the single-rounding exp and p = e * RN(1 / den): 5% faster at
// the headline than the compensated exp with the correctly rounded e / den
// (CSA_BWD_SMALL_EXP=softmax_exp, CSA_BWD_SMALL_DIV_RN=1), for 0.0012%
// instead of 0.0008% of dkv and 0.0045% instead of 0.0040% of dscore
// differing from the oracle by one bf16 step; neither reaches bit identity.
#ifndef CSA_BWD_SMALL_EXP
#define CSA_BWD_SMALL_EXP softmax_exp_fast
#endif
// 1: windows of up to 4 slots load the next row's inputs before computing the
// current row (0: one row at a time). Measured at ratio 2, coff 2, d 128
// (62766 ragged tokens): 33.4 us against 36.5 us with L2 clean, 38.6 against
// 41.2 us after a write flush.
#ifndef CSA_BWD_PREFETCH
#define CSA_BWD_PREFETCH 1
#endif
constexpr bool kBwdPrefetch = CSA_BWD_PREFETCH != 0;
#ifndef CSA_BWD_SMALL_DIV_RN
#define CSA_BWD_SMALL_DIV_RN 0
#endif
constexpr int kCv = 4;  // columns per thread (8-byte vectors)


// Small window (W <= 8): blockDim = (TX, TY); a thread owns 4 consecutive
// columns (8-byte vectors) of one row at a time, rows strided by the grid.
// D > 0 fixes head_dim at compile time (slot offsets become immediates);
// D == 0 reads it from the problem.
template <int R, int COFF, int D>
__global__ void __launch_bounds__(kThreads, 2)
bwd_small_kernel(const BwdParams bp) {
  grid_dependency_wait();
  allow_dependent_launch();
  constexpr int W = COFF * R;
  using S = Slot<R, COFF>;
  const Problem& p = bp.p;
  const int d = D > 0 ? D : p.d;
  const int TX = blockDim.x, TY = blockDim.y;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int tid = ty * TX + tx, nthr = TX * TY;
  const int ncv = d / kCv;
  const int cv = blockIdx.x * TX + tx;
  const bool col_ok = cv < ncv;
  const int64_t ld = (int64_t)COFF * d;
  const int j0 = cv * kCv;
  const int tile_cols = TX * kCv;
  // element offset of slot k from (row base token, column j0)
  auto koff = [&](int k) -> int64_t { return (S::tok(0, k)) * ld + S::half(k) * d; };

  // [W][tile_cols]: the APE slice of this column tile, later the dape combine
  // buffer; then the segment arrays (seg_smem_bytes)
  extern __shared__ float sm[];
  for (int i = tid; i < W * tile_cols; i += nthr) {
    const int k = i / tile_cols;
    const int col = blockIdx.x * tile_cols + (i - k * tile_cols);
    sm[i] = col < d ? __ldg(p.ape + (int64_t)S::ape_row(k) * ld + S::half(k) * d + col) : 0.0f;
  }
  const SegMap sg = stage_segments(p.cu, p.cuc, p.nseq, reinterpret_cast<int32_t*>(sm + W * tile_cols),
                                   tid, nthr);
  __syncthreads();
  const float* ape_s = sm + tx * kCv;

  float dacc[W][kCv];
#pragma unroll
  for (int k = 0; k < W; ++k)
#pragma unroll
    for (int c = 0; c < kCv; ++c) dacc[k][c] = 0.0f;

  const uint2 zero2 = make_uint2(0u, 0u);
  const int64_t true_rows = sg.cuc[p.nseq];
  const int64_t stride = (int64_t)gridDim.y * TY;
  int hint = 0;
  // row b's inputs (a row that breaks the preconditions, or past capacity,
  // reads nothing)
  auto load_row = [&](int64_t b, const RowInfo& ri, uint2 (&kvv)[W], uint2 (&scv)[W], uint2& gv) {
    if (!row_in_bounds<R, COFF>(ri, p.T) || b >= p.C) return;
    const int64_t rowoff = ri.base * ld + j0;
#pragma unroll
    for (int k = 0; k < W; ++k) {
      if (S::masked(ri.first, k)) {
        kvv[k] = zero2;
        scv[k] = make_uint2(kNegInfBf16x2, kNegInfBf16x2);
      } else {
        kvv[k] = ld_stream8(p.kv + rowoff + koff(k));
        scv[k] = ld_stream8(p.score + rowoff + koff(k));
      }
    }
    gv = ld_stream8(bp.grad_out + b * d + j0);
  };
  // row b from its loaded inputs: outputs, dape sums, owned zero positions
  auto run_row = [&](int64_t b, const RowInfo& ri, uint2 (&kvv)[W], uint2 (&scv)[W], const uint2 gv) {
    if (!row_in_bounds<R, COFF>(ri, p.T)) return;  // violated preconditions: skip
    const int64_t rowoff = ri.base * ld + j0;
    uint16_t* dkv_row = bp.dkv + rowoff;
    uint16_t* dsc_row = bp.dscore + rowoff;
    if (b < p.C) {

      // z = score + ape, then in place e = exp(z - m), then p = e * (1 / den)
      float pz[W][kCv];
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const float4 a = *reinterpret_cast<const float4*>(ape_s + k * tile_cols);
        pz[k][0] = add_bf16_f32(bf16_half(scv[k].x, 0), a.x);
        pz[k][1] = add_bf16_f32(bf16_half(scv[k].x, 1), a.y);
        pz[k][2] = add_bf16_f32(bf16_half(scv[k].y, 0), a.z);
        pz[k][3] = add_bf16_f32(bf16_half(scv[k].y, 1), a.w);
      }
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        // both columns of the pair: m, e, den, p, then S
        float sum[2], g[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = 2 * c2 + h;
          float m = pz[0][c];
#pragma unroll
          for (int k = 1; k < W; ++k) m = max_nan(m, pz[k][c]);
          float den = 0.0f;
#pragma unroll
          for (int k = 0; k < W; ++k) {
            pz[k][c] = CSA_BWD_SMALL_EXP(__fsub_rn(pz[k][c], m));
            den = __fadd_rn(den, pz[k][c]);
          }
          const float y = __frcp_rn(den);
#if CSA_BWD_SMALL_DIV_RN
#pragma unroll
          for (int k = 0; k < W; ++k) pz[k][c] = div_rn_by_rcp(pz[k][c], den, y);
#else
#pragma unroll
          for (int k = 0; k < W; ++k) pz[k][c] = __fmul_rn(pz[k][c], y);
#endif
          g[h] = bf16_at(c2 ? gv.y : gv.x, h);
          float acc = 0.0f;
#pragma unroll
          for (int k = 0; k < W; ++k) {
            // RN(g kv) from the bf16 halves (the product is exact)
            const float dp = mul_bf16(bf16_half(c2 ? gv.y : gv.x, h), bf16_half(c2 ? kvv[k].y : kvv[k].x, h));
            acc = __fadd_rn(acc, __fmul_rn(dp, pz[k][c]));
          }
          sum[h] = acc;
        }
        // dscore = p (dp - S), dkv = g p, packed per slot as soon as both columns exist;
        // the packed words reuse the raw score registers, which are dead by now
#pragma unroll
        for (int k = 0; k < W; ++k) {
          float dz[2], dk[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = 2 * c2 + h;
            const float dp = mul_bf16(bf16_half(c2 ? gv.y : gv.x, h), bf16_half(c2 ? kvv[k].y : kvv[k].x, h));
            dz[h] = __fmul_rn(pz[k][c], __fsub_rn(dp, sum[h]));
            dk[h] = __fmul_rn(g[h], pz[k][c]);
            dacc[k][c] = __fadd_rn(dacc[k][c], dz[h]);
          }
          if (c2 == 0) {
            scv[k].x = pack_bf16x2(dz[0], dz[1]);
            kvv[k].x = pack_bf16x2(dk[0], dk[1]);
          } else {
            scv[k].y = pack_bf16x2(dz[0], dz[1]);
            kvv[k].y = pack_bf16x2(dk[0], dk[1]);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < W; ++k) {
        if (S::masked(ri.first, k)) continue;
        st_stream8(dkv_row + koff(k), kvv[k]);
        st_stream8(dsc_row + koff(k), scv[k]);
      }
    } else {
      // a row past capacity has no output slot: zero gradient at its positions
#pragma unroll
      for (int k = 0; k < W; ++k) {
        if (S::masked(ri.first, k)) continue;
        st_stream8(dkv_row + koff(k), zero2);
        st_stream8(dsc_row + koff(k), zero2);
      }
    }
    if (ri.last) {
      // the segment's last row owns its block's unread first-half columns ...
      if (COFF == 2) {
#pragma unroll
        for (int t = 0; t < R; ++t) {
          st_stream8(dkv_row + t * ld, zero2);
          st_stream8(dsc_row + t * ld, zero2);
        }
      }
      // ... and the segment's tail tokens (seqlen % ratio of them)
      const int64_t tail_end = ri.seg_end < p.T ? ri.seg_end : p.T;
      for (int64_t tok = ri.base + R; tok < tail_end; ++tok) {
#pragma unroll
        for (int h = 0; h < COFF; ++h) {
          const int64_t off = tok * ld + h * d + j0;
          st_stream8(bp.dkv + off, zero2);
          st_stream8(bp.dscore + off, zero2);
        }
      }
    }
  };
  int64_t b = (int64_t)blockIdx.y * TY + ty;
  if constexpr (kBwdPrefetch && W <= 4) {
    // windows of up to 4 slots have the registers for the next row's inputs:
    // their loads are in flight while this row computes
    RowInfo ri{};
    uint2 kvv[W], scv[W], gv = zero2;
    if (col_ok && b < true_rows) {
      ri = row_info_from(sg.cu, sg.cuc, p.nseq, b, true_rows, R, hint);
      load_row(b, ri, kvv, scv, gv);
    }
    for (; col_ok && b < true_rows; b += stride) {
      RowInfo rn{};
      uint2 kvn[W], scn[W], gn = zero2;
      if (b + stride < true_rows) {
        rn = row_info_from(sg.cu, sg.cuc, p.nseq, b + stride, true_rows, R, hint);
        load_row(b + stride, rn, kvn, scn, gn);
      }
      run_row(b, ri, kvv, scv, gv);
      ri = rn;
      gv = gn;
#pragma unroll
      for (int k = 0; k < W; ++k) {
        kvv[k] = kvn[k];
        scv[k] = scn[k];
      }
    }
  } else {
    for (; col_ok && b < true_rows; b += stride) {
      const RowInfo ri = row_info_from(sg.cu, sg.cuc, p.nseq, b, true_rows, R, hint);
      uint2 kvv[W], scv[W], gv = zero2;
      load_row(b, ri, kvv, scv, gv);
      run_row(b, ri, kvv, scv, gv);
    }
  }

  zero_orphans(bp, R);

  // combine the TY thread rows in ascending order, then write this CTA's
  // slice of the partial of row group blockIdx.y
  __syncthreads();
  for (int t = 0; t < TY; ++t) {
    if (ty == t && col_ok) {
#pragma unroll
      for (int k = 0; k < W; ++k)
#pragma unroll
        for (int c = 0; c < kCv; ++c) {
          float* s = sm + k * tile_cols + tx * kCv + c;
          *s = t == 0 ? dacc[k][c] : __fadd_rn(*s, dacc[k][c]);
        }
    }
    __syncthreads();
  }
  float* part = bp.partial + (int64_t)blockIdx.y * (R * ld);
  for (int i = tid; i < W * tile_cols; i += nthr) {
    const int k = i / tile_cols;
    const int col = blockIdx.x * tile_cols + (i - k * tile_cols);
    if (col < d) part[(int64_t)S::ape_row(k) * ld + S::half(k) * d + col] = sm[i];
  }
}

// dape[e] = sum over groups g of partial[g][e] in two fixed levels. A lane
// owns 4 consecutive elements (16-byte loads; every group row starts on a
// 32-byte boundary because ratio * coff * d is a multiple of 8); blockDim.x
// lanes cover consecutive element vectors and blockDim.y lanes share each
// vector. Lane y sums groups y, y + Y, y + 2Y, ... in ascending order (loads
// issued 8 at a time so they overlap), then a fixed tree adds the Y lane sums
// (y += y + Y/2, y + Y/4, ...). X and Y are powers of two fixed by the launch
// from n and groups, so the order is the same on every run.
constexpr int kReduceThreads = 1024;
constexpr int kReduceMaxLanes = 64;

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z),
                     __fadd_rn(a.w, b.w));
}

__global__ void __launch_bounds__(kReduceThreads)
dape_reduce_kernel(const float4* __restrict__ partial, int32_t groups, int64_t n4,
                   float4* __restrict__ dape) {
  grid_dependency_wait();
  allow_dependent_launch();
  __shared__ float4 red[kReduceThreads];
  const int X = blockDim.x, Y = blockDim.y;
  const int64_t e = (int64_t)blockIdx.x * X + threadIdx.x;
  float4 s = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (e < n4) {
    for (int g0 = threadIdx.y; g0 < groups; g0 += 8 * Y) {
      float4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int g = g0 + i * Y;
        v[i] = g < groups ? __ldcs(partial + (int64_t)g * n4 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (g0 + i * Y < groups) s = add4(s, v[i]);
    }
  }
  if (Y == 1) {
    if (e < n4) dape[e] = s;
    return;
  }
  float4* mine = red + threadIdx.y * X + threadIdx.x;
  *mine = s;
  for (int h = Y >> 1; h > 0; h >>= 1) {  // Y is uniform over the block
    __syncthreads();
    if (threadIdx.y < h) *mine = add4(*mine, mine[h * X]);
  }
  if (threadIdx.y == 0 && e < n4) dape[e] = *mine;
}

template <int R, int COFF, int D>
cudaError_t plan_small_d(const Problem& p, BwdShape* s) {
  constexpr int W = COFF * R;
  const int ncv = p.d / kCv;
  const int tx = ncv <= 128 ? ncv : 128;
  const int ty = kThreads / tx > 0 ? kThreads / tx : 1;
  const int tiles = (ncv + tx - 1) / tx;
  const size_t smem = sizeof(float) * W * tx * kCv + seg_smem_bytes(p.nseq);
  auto kern = bwd_small_kernel<R, COFF, D>;
  if (cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), 128 * 1024)) return e;
  const int occ = occupancy(reinterpret_cast<const void*>(kern), tx * ty, smem);
  int64_t gy = (int64_t)kGroupingSms * occ / tiles;
  const int64_t row_blocks = (p.C + ty - 1) / ty;
  if (gy > row_blocks) gy = row_blocks;
  if (gy < 1) gy = 1;
  if (gy > 65535) gy = 65535;
  s->grid = dim3(tiles, (unsigned)gy);
  s->block = dim3(tx, ty);
  s->smem = smem;
  s->groups = (int32_t)gy;
  return cudaSuccess;
}

template <int R, int COFF>
cudaError_t plan_small(const Problem& p, BwdShape* s) {
  if (p.d == 512) return plan_small_d<R, COFF, 512>(p, s);
  if (p.d == 128) return plan_small_d<R, COFF, 128>(p, s);
  return plan_small_d<R, COFF, 0>(p, s);
}

template <int R, int COFF>
cudaError_t run_small(const BwdParams& b, const BwdShape& s, cudaStream_t stream) {
  auto kern = b.p.d == 512 ? bwd_small_kernel<R, COFF, 512>
             : b.p.d == 128 ? bwd_small_kernel<R, COFF, 128> : bwd_small_kernel<R, COFF, 0>;
  return launch_dependent(kern, s.grid, s.block, s.smem, stream, b);
}

#define CSA_BWD_SMALL_DISPATCH(FN, ...)                       \
  switch (p.ratio * 4 + p.coff) {                                 \
    case 2 * 4 + 1: return FN<2, 1>(__VA_ARGS__);                 \
    case 2 * 4 + 2: return FN<2, 2>(__VA_ARGS__);                 \
    case 4 * 4 + 1: return FN<4, 1>(__VA_ARGS__);                 \
    case 4 * 4 + 2: return FN<4, 2>(__VA_ARGS__);                 \
    case 8 * 4 + 1: return FN<8, 1>(__VA_ARGS__);                 \
    default: break;                                               \
  }

}  // namespace

cudaError_t plan_bwd(const Problem& p, BwdShape* shape) {
  if (p.exact) return plan_bwd_bitwise(p, shape);
  CSA_BWD_SMALL_DISPATCH(plan_small, p, shape)
  return plan_bwd_long(p, shape);  // windows of 16 slots and more
}

cudaError_t launch_bwd(const BwdParams& b, const BwdShape& shape, cudaStream_t stream) {
  const Problem& p = b.p;
  if (p.exact) return launch_bwd_bitwise(b, shape, stream);
  CSA_BWD_SMALL_DISPATCH(run_small, b, shape, stream)
  return launch_bwd_long(b, shape, stream);
}

cudaError_t launch_dape_reduce(const float* partial, int32_t groups, int64_t n, float* dape,
                               cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int64_t n4 = n / 4;  // n = ratio * coff * d, a multiple of 8
  // Y: lanes per element vector, enough that each issues about one batch of
  // 8 loads; X: element vectors per block, narrower when there are few
  // vectors so that about 128+ blocks share the work. Both follow from the
  // problem (n, groups) alone.
  int lanes = 1;
  while (lanes < kReduceMaxLanes && (int64_t)lanes * 8 < groups) lanes *= 2;
  int x = 32;
  while (x > 4 && (n4 + x - 1) / x < 128) x >>= 1;
  while (x * lanes > kReduceThreads) lanes >>= 1;
  const int64_t blocks = (n4 + x - 1) / x;
  return launch_dependent(dape_reduce_kernel, dim3((unsigned)blocks), dim3(x, lanes), 0, stream,
                          reinterpret_cast<const float4*>(partial), groups, n4,
                          reinterpret_cast<float4*>(dape));
}

}  // namespace csa
