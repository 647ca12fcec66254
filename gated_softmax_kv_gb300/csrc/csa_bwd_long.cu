// Long-window backward (window W = coff * ratio >= 16, e.g. ratio 128) of the
// CSA/HCA fused Compressor for sm_103a; the operation and the ownership of
// every dkv / dscore position are those of csa_bwd.cu (cuDNN-frontend "CSA
// Fused Compressor", sections "Semantics" and "Class API").
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_bwd_common.cuh"
#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

namespace {

// exp of the long-window backward. Windows of 16 slots and more have no
// bitwise target (the page aims at bit identity for ratios 2 and 4 only), so
// the per-element weights take the single-rounding exp (softmax_exp_fast2,
// two lanes at a time) and T = sum (g kv) e one FMA per slot; the chunk
// merges and the rescaling of a chunk to the row max use CSA_BWD_LONG_EXP.
#ifndef CSA_BWD_LONG_EXP
#define CSA_BWD_LONG_EXP softmax_exp_fast
#endif
// Long-window backward: windows of at least this many slots give each warp 16
// slots x 2 columns (8-warp CTAs, two per SM) instead of 8 slots x 4 columns.
// 1: kv / score / grad_out loads skip L1 allocation, so the L1 keeps the APE
// tile the threads re-read every row (ratio 128: 1.3% faster at 131072 tokens,
// coff 1, head_dim 512; 0: streaming loads)
#ifndef CSA_BWD_LONG_NOALLOC
#define CSA_BWD_LONG_NOALLOC 1
#endif
// 1: dkv / dscore stores skip L1 allocation too and keep the normal L2 policy
// (ratio 128: 2.3% faster backward at 131072 tokens, coff 1, head_dim 512;
// 0: evict-first stores)
#ifndef CSA_BWD_LONG_NOALLOC_ST
#define CSA_BWD_LONG_NOALLOC_ST 1
#endif
#ifndef CSA_BWD_LONG_KPT16_FROM
#define CSA_BWD_LONG_KPT16_FROM 128
#endif

// Long window (W >= 16): blockDim = (32, NCH) with NCH = W / KPT (KPT = 8
// slots per warp, 16 for W = 256). Warp y owns window slots
// [KPT y, KPT y + KPT) and lane l owns VC consecutive columns of a
// (32 VC)-column tile (blockIdx.x), so every load and store of a warp covers
// 32 VC * 2 contiguous bytes of one token row. The CTA walks rows
// b = blockIdx.y, blockIdx.y + gridDim.y, ... and per row:
//   phase 1  z = score + ape, the chunk's max m_c, e = exp(z - m_c), sum e and
//            T_c = sum (g kv) e
//   merge    (max, sum, T) of the NCH chunks of a column, in a fixed order:
//            NCH/VC threads take VC chunks each, then a butterfly over those
//            lanes (commutative combines, so every lane gets the same bits);
//            S = sum (g kv) p = T / den
//   phase 2  p = e * (exp(m_c - M) / den) (one exp and one reciprocal per
//            column and chunk), dscore = p (g kv - S), dkv = g p, stores; dape
//            accumulates in shared memory (each thread owns KPT slots x VC
//            columns of the [W][TC] table, so no barrier guards it)
// Two barriers per row. The next row's kv, score and grad_out loads are
// issued before the merge, so they are in flight through the merge and
// phase 2 (one CTA of NCH warps per SM would otherwise leave HBM idle while
// it computes).
template <int W>
struct LongShape {
  static constexpr int kKpt = W >= CSA_BWD_LONG_KPT16_FROM ? 16 : 8;                   // slots per warp
  static constexpr int kVc = (W >= CSA_BWD_LONG_KPT16_FROM || W <= 16) ? 2 : 4;        // columns per lane
  static constexpr int kNch = W / kKpt;                      // warps per CTA
  static constexpr int kThreads = 32 * kNch;
  static constexpr int kMinBlocks = kThreads >= 512 ? 1 : 512 / kThreads;  // <= 128 registers
  static_assert(kNch % kVc == 0, "each column's chunks split evenly over its merge threads");
};

template <int VC>
struct ColVec;
template <>
struct ColVec<2> {
  using T = uint32_t;
#if CSA_BWD_LONG_NOALLOC
  static __device__ __forceinline__ T load(const uint16_t* p) {
    uint32_t v;
    asm("ld.global.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
  }
#else
  static __device__ __forceinline__ T load(const uint16_t* p) { return __ldcs(reinterpret_cast<const uint32_t*>(p)); }
#endif
#if CSA_BWD_LONG_NOALLOC_ST
  static __device__ __forceinline__ void store(uint16_t* p, T v) {
    asm volatile("st.global.L1::no_allocate.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
  }
#else
  static __device__ __forceinline__ void store(uint16_t* p, T v) { __stcs(reinterpret_cast<uint32_t*>(p), v); }
#endif
  static __device__ __forceinline__ float elem(T v, int c) { return bf16_at(v, c); }
  static __device__ __forceinline__ uint16_t half(T v, int c) { return bf16_half(v, c); }
  static __device__ __forceinline__ T zero() { return 0u; }
  static __device__ __forceinline__ T ninf() { return kNegInfBf16x2; }
  static __device__ __forceinline__ T pack(const float* x) { return pack_bf16x2(x[0], x[1]); }
  // VC consecutive floats of shared memory (8-byte aligned)
  static __device__ __forceinline__ void load_f(const float* p, float* x) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x;
    x[1] = v.y;
  }
  static __device__ __forceinline__ void store_f(float* p, const float* x) {
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
  }
  static __device__ __forceinline__ void add_f(float* p, const float* x) {
    float2 v = *reinterpret_cast<float2*>(p);
    v.x = __fadd_rn(v.x, x[0]);
    v.y = __fadd_rn(v.y, x[1]);
    *reinterpret_cast<float2*>(p) = v;
  }
};
template <>
struct ColVec<4> {
  using T = uint2;
#if CSA_BWD_LONG_NOALLOC
  static __device__ __forceinline__ T load(const uint16_t* p) {
    uint2 v;
    asm("ld.global.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
  }
#else
  static __device__ __forceinline__ T load(const uint16_t* p) { return ld_stream8(p); }
#endif
  static __device__ __forceinline__ void store(uint16_t* p, T v) { st_stream8(p, v); }
  static __device__ __forceinline__ float elem(T v, int c) { return bf16_at(c < 2 ? v.x : v.y, c & 1); }
  static __device__ __forceinline__ uint16_t half(T v, int c) { return bf16_half(c < 2 ? v.x : v.y, c & 1); }
  static __device__ __forceinline__ T zero() { return make_uint2(0u, 0u); }
  static __device__ __forceinline__ T ninf() { return make_uint2(kNegInfBf16x2, kNegInfBf16x2); }
  static __device__ __forceinline__ T pack(const float* x) {
    return make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
  }
  // VC consecutive floats of shared memory (16-byte aligned)
  static __device__ __forceinline__ void load_f(const float* p, float* x) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x;
    x[1] = v.y;
    x[2] = v.z;
    x[3] = v.w;
  }
  static __device__ __forceinline__ void store_f(float* p, const float* x) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  }
  static __device__ __forceinline__ void add_f(float* p, const float* x) {
    float4 v = *reinterpret_cast<float4*>(p);
    v.x = __fadd_rn(v.x, x[0]);
    v.y = __fadd_rn(v.y, x[1]);
    v.z = __fadd_rn(v.z, x[2]);
    v.w = __fadd_rn(v.w, x[3]);
    *reinterpret_cast<float4*>(p) = v;
  }
};

// fixed-order merge of (max, sum exp, sum (g kv) exp) triples rescaled to the
// common max: m = max, s = s_a e^(m_a - m) + s_b e^(m_b - m), t likewise.
// Symmetric in a and b, so both lanes of a butterfly step get the same bits.
__device__ __forceinline__ void merge_max_sum2(float& m, float& s, float& t, float mb, float sb,
                                               float tb) {
  const float kNegInf = __int_as_float(0xff800000);
  const float mn = max_nan(m, mb);
  const float mu = mn == kNegInf ? 0.0f : mn;
  const float fa = CSA_BWD_LONG_EXP(__fsub_rn(m, mu)), fb = CSA_BWD_LONG_EXP(__fsub_rn(mb, mu));
  s = __fadd_rn(__fmul_rn(s, fa), __fmul_rn(sb, fb));
  t = __fadd_rn(__fmul_rn(t, fa), __fmul_rn(tb, fb));
  m = mn;
}

// D > 0 fixes head_dim at compile time (slot offsets become immediates);
// D == 0 reads it from the problem.
template <int R, int COFF, int D>
__global__ void __launch_bounds__(LongShape<COFF * R>::kThreads, LongShape<COFF * R>::kMinBlocks)
bwd_long_kernel(const BwdParams bp) {
  grid_dependency_wait();
  allow_dependent_launch();
  constexpr int W = COFF * R;
  constexpr int KPT = LongShape<W>::kKpt;
  constexpr int VC = LongShape<W>::kVc;
  constexpr int NCH = LongShape<W>::kNch;
  constexpr int NT = LongShape<W>::kThreads;
  constexpr int TC = 32 * VC;      // tile columns
  constexpr int G = NCH / VC;      // merge threads per column
  constexpr int LDS = TC + 1;      // padded row stride of the chunk tables
  using S = Slot<R, COFF>;
  using V = ColVec<VC>;
  const Problem& p = bp.p;
  const int d = D > 0 ? D : p.d;
  const int lane = threadIdx.x, y = threadIdx.y;
  const int tid = y * 32 + lane;
  const int ncv = d / VC;
  const int cv = blockIdx.x * 32 + lane;
  const bool col_ok = cv < ncv;
  const int64_t ld = (int64_t)COFF * d;
  const int j0 = cv * VC;
  const int k0 = y * KPT;
  const float kNegInf = __int_as_float(0xff800000);

  __shared__ float m_s[NCH * LDS], d_s[NCH * LDS], s_s[NCH * LDS];
  __shared__ float M_s[TC], D_s[TC], S_s[TC];
  // dape sums of the tile, [W][TC] (each cell belongs to one thread), then
  // the segment arrays (seg_smem_bytes)
  extern __shared__ __align__(16) float dacc_s[];
  float* dacc_t = dacc_s + k0 * TC + lane * VC;  // 8 (VC 2) or 16 (VC 4) byte aligned
#pragma unroll
  for (int t = 0; t < KPT; ++t) {
    const float z[VC] = {};
    V::store_f(dacc_t + t * TC, z);
  }

  // this thread's APE values (slots k0.., columns j0..) are re-read per row through L1
  const float* ape_t = p.ape + (int64_t)S::ape_row(k0) * ld + S::half(k0) * d + j0;

  // merge thread layout: column mc of the tile, group member mq (G per column)
  const int mc = tid / G, mq = tid % G;

  // The next row's kv, score and grad_out are loaded while the current row
  // merges and runs phase 2 (score into the registers phase 1 has consumed).
  typename V::T kvw[KPT], scw[KPT], gw = V::zero();
  auto offset = [&](const RowInfo& r) {
    return r.base * ld + S::tok(0, k0) * ld + S::half(k0) * d + j0;
  };
  auto loads = [&](int64_t rb, const RowInfo& r, typename V::T (&kvb)[KPT], typename V::T& gb) {
    // rows past capacity and rows that break the preconditions load nothing
    if (rb >= p.C || !row_in_bounds<R, COFF>(r, p.T)) {
#pragma unroll
      for (int t = 0; t < KPT; ++t) kvb[t] = V::zero();
      return;
    }
    const bool act = col_ok && !S::masked(r.first, k0);
    const int64_t off = offset(r);
#pragma unroll
    for (int t = 0; t < KPT; ++t) {
      kvb[t] = act ? V::load(p.kv + off + t * ld) : V::zero();
      scw[t] = act ? V::load(p.score + off + t * ld) : V::ninf();
    }
    gb = col_ok ? V::load(bp.grad_out + rb * d + j0) : V::zero();
  };

  // the segment arrays after the dape table, in shared memory when they fit
  const SegMap sg = stage_segments(p.cu, p.cuc, p.nseq, reinterpret_cast<int32_t*>(dacc_s + W * TC),
                                   tid, NT);
  __syncthreads();
  const int64_t true_rows = sg.cuc[p.nseq];
  int64_t b = blockIdx.y;
  RowInfo ri{};
  int hint = 0;  // segment of the last row looked up (rows only increase)
  if (b < true_rows) {
    ri = row_info_from(sg.cu, sg.cuc, p.nseq, b, true_rows, R, hint);
    loads(b, ri, kvw, gw);
  }
  for (; b < true_rows;) {
    const bool row_ok = row_in_bounds<R, COFF>(ri, p.T);  // uniform over the CTA
    const bool active = col_ok && !S::masked(ri.first, k0);
    const int64_t off = offset(ri);
    const bool compute = row_ok && b < p.C;  // uniform over the CTA
    float g[VC], mloc[VC];
    float pz[KPT][VC];
    if (compute) {
#pragma unroll
      for (int c = 0; c < VC; ++c) g[c] = V::elem(gw, c);
#pragma unroll
      for (int t = 0; t < KPT; ++t) {
#pragma unroll
        for (int c = 0; c < VC; c += 2) {
          const float2 a = col_ok ? __ldg(reinterpret_cast<const float2*>(ape_t + t * ld + c))
                                  : make_float2(0.0f, 0.0f);
          const float2 z = make_float2(add_bf16_f32(V::half(scw[t], c), a.x),
                                       add_bf16_f32(V::half(scw[t], c + 1), a.y));
          pz[t][c] = z.x;
          pz[t][c + 1] = z.y;
        }
      }
      // phase 1: per column, the chunk's max m_c, e = exp(z - m_c), its sum
      // and T_c = sum (g kv) e; one fixed-order merge of (max, sum, T) then
      // gives the row's max M, den and S = T / den together. Columns go in
      // pairs through the two-lane fp32 instructions (same roundings).
#pragma unroll
      for (int c = 0; c < VC; c += 2) {
        // the chunk's max per column (three-input max, NaN propagating)
        const float m0 = max_range<0, KPT>([&](int t) { return pz[t][c]; });
        const float m1 = max_range<0, KPT>([&](int t) { return pz[t][c + 1]; });
        // an all -inf chunk contributes 0
        const float2 mu = make_float2(m0 == kNegInf ? 0.0f : m0, m1 == kNegInf ? 0.0f : m1);
        const float2 g2 = make_float2(g[c], g[c + 1]);
        float2 sum = make_float2(0.0f, 0.0f), tsum = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int t = 0; t < KPT; ++t) {
          const float2 e = softmax_exp_fast2(sub2_rn(make_float2(pz[t][c], pz[t][c + 1]), mu));
          pz[t][c] = e.x;
          pz[t][c + 1] = e.y;
          sum = add2_rn(sum, e);
          // dp = RN(g kv) from the bf16 halves (exact products)
          const float2 dp = make_float2(mul_bf16(V::half(gw, c), V::half(kvw[t], c)),
                                        mul_bf16(V::half(gw, c + 1), V::half(kvw[t], c + 1)));
          tsum = fma2_rn(dp, e, tsum);
        }
        mloc[c] = m0;
        mloc[c + 1] = m1;
        m_s[y * LDS + lane * VC + c] = m0;
        m_s[y * LDS + lane * VC + c + 1] = m1;
        d_s[y * LDS + lane * VC + c] = sum.x;
        d_s[y * LDS + lane * VC + c + 1] = sum.y;
        s_s[y * LDS + lane * VC + c] = tsum.x;
        s_s[y * LDS + lane * VC + c + 1] = tsum.y;
      }
    }
    // prefetch the next row of this CTA
    const int64_t bn = b + gridDim.y;
    RowInfo rn{};
    typename V::T kvn[KPT], gn = V::zero();
    if (bn < true_rows) {
      rn = row_info_from(sg.cu, sg.cuc, p.nseq, bn, true_rows, R, hint);
      loads(bn, rn, kvn, gn);
    }
    if (compute) {
      __syncthreads();
      {
        float m = m_s[(mq * VC) * LDS + mc], sm = d_s[(mq * VC) * LDS + mc];
        float tm = s_s[(mq * VC) * LDS + mc];
#pragma unroll
        for (int i = 1; i < VC; ++i)
          merge_max_sum2(m, sm, tm, m_s[(mq * VC + i) * LDS + mc], d_s[(mq * VC + i) * LDS + mc],
                         s_s[(mq * VC + i) * LDS + mc]);
#pragma unroll
        for (int mask = 1; mask < G; mask <<= 1)
          merge_max_sum2(m, sm, tm, __shfl_xor_sync(0xffffffffu, m, mask),
                         __shfl_xor_sync(0xffffffffu, sm, mask), __shfl_xor_sync(0xffffffffu, tm, mask));
        if (mq == 0) {
          M_s[mc] = m;
          D_s[mc] = sm;
          S_s[mc] = __fdiv_rn(tm, sm);
        }
      }
      __syncthreads();
      // phase 2: p = e exp(m_c - M) / den, dscore = p (g kv - S), dkv = g p
      float fy[VC], Sv[VC];
#pragma unroll
      for (int c = 0; c < VC; ++c) {
        const float M = M_s[lane * VC + c];
        const float den = D_s[lane * VC + c];
        const float mu = M == kNegInf ? 0.0f : M;
        const float ml = mloc[c] == kNegInf ? 0.0f : mloc[c];
        const float f = CSA_BWD_LONG_EXP(__fsub_rn(ml, mu));  // rescales this chunk's e to the row max
        // one scale per column and chunk: f / den (no per-element division;
        // like the exp above, not correctly rounded)
        fy[c] = __fmul_rn(f, __frcp_rn(den));
        Sv[c] = S_s[lane * VC + c];
      }
#pragma unroll
      for (int t = 0; t < KPT; ++t) {
        float dz[VC], dk[VC];
#pragma unroll
        for (int c = 0; c < VC; c += 2) {
          // dp = RN(g kv) as bf16-input FMAs (no later step can fuse them),
          // so dp - S runs on the two-lane subtraction
          const float2 g2 = make_float2(g[c], g[c + 1]);
          const float2 pp = mul2_rn(make_float2(pz[t][c], pz[t][c + 1]), make_float2(fy[c], fy[c + 1]));
          const float2 dp = make_float2(mul_bf16(V::half(gw, c), V::half(kvw[t], c)),
                                        mul_bf16(V::half(gw, c + 1), V::half(kvw[t], c + 1)));
          const float2 diff = sub2_rn(dp, make_float2(Sv[c], Sv[c + 1]));
          const float2 z = mul2_rn(pp, diff);
          const float2 k = mul2_rn(g2, pp);
          dz[c] = z.x;
          dz[c + 1] = z.y;
          dk[c] = k.x;
          dk[c + 1] = k.y;
        }
        V::add_f(dacc_t + t * TC, dz);
        if (active) {
          V::store(bp.dkv + off + t * ld, V::pack(dk));
          V::store(bp.dscore + off + t * ld, V::pack(dz));
        }
      }
    } else if (row_ok && active) {
      // a row past capacity has no output slot: zero gradient at its positions
#pragma unroll
      for (int t = 0; t < KPT; ++t) {
        V::store(bp.dkv + off + t * ld, V::zero());
        V::store(bp.dscore + off + t * ld, V::zero());
      }
    }
    if (row_ok && ri.last) {
      // unread positions owned by the segment's last row, for this column tile:
      // its block's first-half columns (coff 2) and the segment tail
      const int64_t tail_end = ri.seg_end < p.T ? ri.seg_end : p.T;
      const int64_t n_first = COFF == 2 ? (int64_t)R * 32 : 0;
      const int64_t n_tail = (tail_end - (ri.base + R)) * COFF * 32;
      for (int64_t i = tid; i < n_first + n_tail; i += NT) {
        int64_t tok;
        int h, x;
        if (i < n_first) {
          tok = ri.base + i / 32;
          h = 0;
          x = (int)(i % 32);
        } else {
          const int64_t q = i - n_first;
          tok = ri.base + R + q / (COFF * 32);
          h = (int)((q / 32) % COFF);
          x = (int)(q % 32);
        }
        const int col_v = blockIdx.x * 32 + x;
        if (col_v >= ncv) continue;
        V::store(bp.dkv + tok * ld + h * d + col_v * VC, V::zero());
        V::store(bp.dscore + tok * ld + h * d + col_v * VC, V::zero());
      }
    }
    b = bn;
    ri = rn;
    gw = gn;
#pragma unroll
    for (int t = 0; t < KPT; ++t) kvw[t] = kvn[t];
  }

  zero_orphans(bp, R);

  // each (slot, column) of the tile belongs to exactly one thread
  if (col_ok) {
    float* part = bp.partial + (int64_t)blockIdx.y * (R * ld) + (int64_t)S::ape_row(k0) * ld +
                  S::half(k0) * d + j0;
#pragma unroll
    for (int t = 0; t < KPT; ++t) {
      float v[VC];
      V::load_f(dacc_t + t * TC, v);
#pragma unroll
      for (int c = 0; c < VC; c += 2)
        *reinterpret_cast<float2*>(part + t * ld + c) = make_float2(v[c], v[c + 1]);
    }
  }
}

template <int R, int COFF, int D>
cudaError_t plan_long_d(const Problem& p, BwdShape* s) {
  constexpr int W = COFF * R;
  constexpr int NT = LongShape<W>::kThreads;
  const int ncv = p.d / LongShape<W>::kVc;
  const int tiles = (ncv + 31) / 32;
  auto kern = bwd_long_kernel<R, COFF, D>;
  // dape sums of the tile, then the segment arrays
  const size_t smem = sizeof(float) * W * 32 * LongShape<W>::kVc + seg_smem_bytes(p.nseq);
  // the attribute is set once per kernel: the largest size any problem needs
  constexpr size_t smem_max = sizeof(float) * W * 32 * LongShape<W>::kVc + kSegSmemBytesMax;
  if (cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), (int)smem_max)) return e;
  const int occ = occupancy(reinterpret_cast<const void*>(kern), NT, smem);
  int64_t gy = (int64_t)kGroupingSms * occ / tiles;
  if (gy > p.C) gy = p.C;
  if (gy < 1) gy = 1;
  // even out the rows per CTA
  if (p.C > 0) {
    const int64_t passes = (p.C + gy - 1) / gy;
    gy = (p.C + passes - 1) / passes;
  }
  if (gy > 65535) gy = 65535;
  s->grid = dim3(tiles, (unsigned)gy);
  s->block = dim3(32, LongShape<W>::kNch);
  s->smem = smem;
  s->groups = (int32_t)gy;
  return cudaSuccess;
}

template <int R, int COFF>
cudaError_t plan_long(const Problem& p, BwdShape* s) {
  if (p.d == 512) return plan_long_d<R, COFF, 512>(p, s);
  if (p.d == 128) return plan_long_d<R, COFF, 128>(p, s);
  return plan_long_d<R, COFF, 0>(p, s);
}

template <int R, int COFF>
cudaError_t run_long(const BwdParams& b, const BwdShape& s, cudaStream_t stream) {
  auto kern = b.p.d == 512 ? bwd_long_kernel<R, COFF, 512>
             : b.p.d == 128 ? bwd_long_kernel<R, COFF, 128> : bwd_long_kernel<R, COFF, 0>;
  return launch_dependent(kern, s.grid, s.block, s.smem, stream, b);
}

#define CSA_BWD_LONG_DISPATCH(FN, ...)                        \
  switch (p.ratio * 4 + p.coff) {                                 \
    case 8 * 4 + 2: return FN<8, 2>(__VA_ARGS__);                 \
    case 16 * 4 + 1: return FN<16, 1>(__VA_ARGS__);               \
    case 16 * 4 + 2: return FN<16, 2>(__VA_ARGS__);               \
    case 32 * 4 + 1: return FN<32, 1>(__VA_ARGS__);               \
    case 32 * 4 + 2: return FN<32, 2>(__VA_ARGS__);               \
    case 64 * 4 + 1: return FN<64, 1>(__VA_ARGS__);               \
    case 64 * 4 + 2: return FN<64, 2>(__VA_ARGS__);               \
    case 128 * 4 + 1: return FN<128, 1>(__VA_ARGS__);             \
    case 128 * 4 + 2: return FN<128, 2>(__VA_ARGS__);             \
    default: return cudaErrorInvalidValue;                        \
  }

}  // namespace

cudaError_t plan_bwd_long(const Problem& p, BwdShape* shape) {
  CSA_BWD_LONG_DISPATCH(plan_long, p, shape)
}

cudaError_t launch_bwd_long(const BwdParams& b, const BwdShape& shape, cudaStream_t stream) {
  const Problem& p = b.p;
  CSA_BWD_LONG_DISPATCH(run_long, b, shape, stream)
}

}  // namespace csa
