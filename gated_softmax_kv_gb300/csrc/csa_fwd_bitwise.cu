// Bitwise forward of the CSA/HCA fused Compressor for windows of W <= 8 slots
// (sm_103a): csa_compress_fwd_exact.
//
// cuDNN-frontend "CSA Fused Compressor", sections "Semantics" and "Numerics":
// out carries the bits of the fp32 eager-order reference of this library --
// z_k = score_k + ape_k, m = max z, e_k = exp(z_k - m) correctly rounded,
// den = sum e (slot order), p_k = e_k / den (IEEE), out = sum_k RN(p_k kv_k)
// in slot order from +0, one bf16 rounding -- while keeping the streaming
// arithmetic for almost every output.
//
// Per (row, column) the kernel
//  1. runs the fast arithmetic: e = ex2.approx(RN(x log2 e)), p = e RN(1/den)
//     and the reference's pooled sum acc = sum RN(p_k kv_k) in slot order
//     with those weights;
//  2. encloses the reference's pooled sum exactly as the bitwise backward
//     encloses its S (csa_bwd_bitwise.cu): with rho_own and rho_com the
//     weights' per-slot and column-common relative bounds (softmax_exp_fast's
//     envelope, both sides' den rounding through the sum of den's partial
//     sums, the product and quotient roundings),
//       acc_ref in [acc - sigma, acc + sigma],
//       sigma = (rho_own + 2^-23) A + rho_com |acc| + 2^-23 P,
//     A = sum |RN(p_k kv_k)|, P = sum of |acc's partial sums| (the kv values
//     are the reference's own, so each term's only uncertainty is p);
//  3. accepts bf16(acc) when RD(acc - sigma) and RU(acc + sigma) round to the
//     same bf16 bits (then so does acc_ref, which lies between them) and the
//     column is in the range the bounds cover (tau <= kTMax, A finite);
//  4. otherwise queues the column (its window copied out of the row buffer,
//     its output offset) in a per-warp shared-memory queue of 64 / W
//     columns. A full queue, and at the end what is left in it, takes one
//     exact pass that overwrites the fast outputs: W / 2 lanes per column,
//     two window slots a lane (correctly rounded exp, correctly rounded
//     division, den and the pooled sum in slot order, summed by every lane
//     of the column from gathered values). About 0.3% of the columns fail
//     at ratio 4, coff 2, head_dim 512, so a pass comes every ~20 rows of a
//     warp instead of a nearly empty one in a third of the rows.
// Rows arrive in a per-warp shared-memory buffer by cp.async one row ahead of
// their computation. A row whose window leaves [0, total_tokens) (violated
// caller preconditions) gets NaN and reads nothing.
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_bitwise.cuh"
#include "csa_device.cuh"
#include "csa_exp_cr.cuh"
#include "csa_internal.h"

namespace csa {

namespace {

constexpr int kThreads = 256;
using namespace bitwise;

// blockDim = (TX, TY) with TX a multiple of 32, so that a warp lies in one
// row; a thread owns 4 consecutive columns (8-byte words) of one row at a
// time, rows strided by the grid. D > 0 fixes head_dim at compile time.
template <int R, int COFF, int D>
__global__ void __launch_bounds__(kThreads, 2)
fwd_bitwise_kernel(const FwdParams f) {
  grid_dependency_wait();
  allow_dependent_launch();
  constexpr int W = COFF * R;
  constexpr int L = W / 2;   // lanes per column in the exact pass
  constexpr int P = 32 / L;  // columns per exact pass
  using S = Slot<R, COFF>;
  using B = Bounds<W>;
  const Problem& p = f.p;
  const int d = D > 0 ? D : p.d;
  const int TX = blockDim.x, TY = blockDim.y;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int tid = ty * TX + tx, nthr = TX * TY;
  const int lane = tid & 31;
  const int ncv = d / kCv;
  const int cv = blockIdx.x * TX + tx;
  const bool col_ok = cv < ncv;
  const int64_t ld = (int64_t)COFF * d;
  const int j0 = cv * kCv;
  const int tile_cols = TX * kCv;
  auto koff = [&](int k) -> int64_t { return (S::tok(0, k)) * ld + S::half(k) * d; };

  // [W][tile_cols] APE slice, then two row buffers per warp (the current row
  // and the next one, in flight), then the warps' queues of undecided
  // columns, then the segment arrays (seg_smem_bytes)
  extern __shared__ float sm[];
  __shared__ float tab[2 * kExpTableSize];
  exp_cr_table(tab);
  for (int i = tid; i < W * tile_cols; i += nthr) {
    const int k = i / tile_cols;
    const int col = blockIdx.x * tile_cols + (i - k * tile_cols);
    sm[i] = col < d ? __ldg(p.ape + (int64_t)S::ape_row(k) * ld + S::half(k) * d + col) : 0.0f;
  }
  RowBuf<W>* const rb0 = reinterpret_cast<RowBuf<W>*>(sm + W * tile_cols);
  RowBuf<W>* rbs = rb0 + 2 * (tid >> 5);
  Pending<W>* const pq0 = reinterpret_cast<Pending<W>*>(rb0 + 2 * (nthr >> 5));
  Pending<W>& pq = pq0[tid >> 5];
  const SegMap sg = stage_segments(p.cu, p.cuc, p.nseq, reinterpret_cast<int32_t*>(pq0 + (nthr >> 5)),
                                   tid, nthr);
  __syncthreads();
  const float* ape_s = sm + tx * kCv;
  constexpr int kCap = Pending<W>::kCap;
  static_assert(kCap == P, "a pass takes the whole queue");

  const uint2 zero2 = make_uint2(0u, 0u);
  const int64_t true_rows = sg.cuc[p.nseq];
  const int64_t stride = (int64_t)gridDim.y * TY;
  const uint32_t lt = (1u << lane) - 1u;
  int hint = 0;

  // The window of row `row` into `buf`: asynchronous copies of kv and score
  // (constants for masked slots and lanes without columns); rows that break
  // the preconditions copy nothing.
  auto fetch = [&](const RowInfo& info, RowBuf<W>& buf) {
    if (!row_in_bounds<R, COFF>(info, p.T)) return;
    const int64_t off = info.base * ld + j0;
#pragma unroll
    for (int k = 0; k < W; ++k) {
      if (S::masked(info.first, k) || !col_ok) {
        buf.kv[k][lane] = zero2;
        buf.sc[k][lane] = make_uint2(kNegInfBf16x2, kNegInfBf16x2);
      } else {
        cp_async8(&buf.kv[k][lane], p.kv + off + koff(k));
        cp_async8(&buf.sc[k][lane], p.score + off + koff(k));
      }
    }
  };

  // The exact pass over the first cnt queued columns: W / 2 lanes a column,
  // two window slots a lane (correctly rounded exp and division), den and the
  // pooled sum in slot order, summed by every lane of the column's group
  // from gathered values (independent shuffles).
  auto exact_pass = [&](int cnt) {
    const int q = lane / L, l = lane % L, gbase = lane & ~(L - 1);
    __syncwarp();
    const bool act = q < cnt;
    const int qe = act ? q : 0;
    const uint32_t sw = lds_u32(&pq.sc[qe][2 * l]);  // slots 2 l and 2 l + 1
    const uint32_t kw = lds_u32(&pq.kv[qe][2 * l]);
    const int tcol = pq.tcol[qe];
    const float2 z = make_float2(__fadd_rn(bf16_lo(sw), sm[(2 * l) * tile_cols + tcol]),
                                 __fadd_rn(bf16_hi(sw), sm[(2 * l + 1) * tile_cols + tcol]));
    float mx = max_nan(z.x, z.y);
#pragma unroll
    for (int o = 1; o < L; o <<= 1) mx = max_nan(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float2 ex = exp_cr2(sub2_rn(z, make_float2(mx, mx)), tab);
    float den = 0.0f;
#pragma unroll
    for (int k = 0; k < W; ++k)
      den = __fadd_rn(den, __shfl_sync(0xffffffffu, (k & 1) ? ex.y : ex.x, gbase + k / 2));
    const float yd = __frcp_rn(den);
    const float2 pw = div2_cr(ex, make_float2(den, den), make_float2(-den, -den),
                              make_float2(yd, yd));
    const float t0 = __fmul_rn(pw.x, bf16_lo(kw)), t1 = __fmul_rn(pw.y, bf16_hi(kw));
    float acc = 0.0f;
#pragma unroll
    for (int k = 0; k < W; ++k)
      acc = __fadd_rn(acc, __shfl_sync(0xffffffffu, (k & 1) ? t1 : t0, gbase + k / 2));
    if (act && l == 0) st_u16(f.out + pq.off[qe], bf16_bits_rn(acc));
    __syncwarp();
  };
  int pend = 0;  // queued columns

  // every lane of a warp runs every row of its warp (the exact pass is warp-wide)
  int64_t b = (int64_t)blockIdx.y * TY + ty;
  if (b < p.C) fetch(row_info_from(sg.cu, sg.cuc, p.nseq, b, true_rows, R, hint), rbs[0]);
  cp_async_commit();
  for (int it = 0; b < p.C; ++it, b += stride) {
    const RowInfo cur = row_info_from(sg.cu, sg.cuc, p.nseq, b, true_rows, R, hint);
    __syncwarp();
    if (b + stride < p.C)
      fetch(row_info_from(sg.cu, sg.cuc, p.nseq, b + stride, true_rows, R, hint), rbs[(it + 1) & 1]);
    cp_async_commit();
    cp_async_wait<1>();  // this row's copies have landed ...
    __syncwarp();        // ... for every lane of the warp
    RowBuf<W>& rb = rbs[it & 1];
    uint16_t* dst = f.out + b * d + j0;
    if (!row_in_bounds<R, COFF>(cur, p.T)) {  // violated preconditions: NaN, no access
      if (col_ok) st_stream8(dst, make_uint2(0x7FC07FC0u, 0x7FC07FC0u));
      continue;
    }
    uint32_t ow[2];
    uint32_t fbits = 0;  // bit 2 c2 + h: column 2 c2 + h left undecided
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
      // the column pair (2 c2, 2 c2 + 1) in the two lanes of f32x2 values
      float2 pz[W];
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const float2 a = *reinterpret_cast<const float2*>(ape_s + k * tile_cols + 2 * c2);
        const uint32_t w = lds_u32(reinterpret_cast<const uint32_t*>(&rb.sc[k][lane]) + c2);
        uint16_t s0, s1;
        split_bf16x2(w, s0, s1);
        pz[k] = make_float2(add_bf16_f32(s0, a.x), add_bf16_f32(s1, a.y));
      }
      auto zx = [&](int k) { return pz[k].x; };
      auto zy = [&](int k) { return pz[k].y; };
      const float2 m = make_float2(max_range<0, W>(zx), max_range<0, W>(zy));
      // smallest logit over the valid slots (fminf skips NaN; m carries it)
      constexpr int kLoValid = COFF == 2 ? R : 0;  // first slot valid on every row
      float2 zmin = make_float2(min_range<kLoValid, W>(zx), min_range<kLoValid, W>(zy));
      if (COFF == 2 && !cur.first)
        zmin = make_float2(fminf(zmin.x, min_range<0, (COFF == 2 ? R : 1)>(zx)),
                           fminf(zmin.y, min_range<0, (COFF == 2 ? R : 1)>(zy)));
      const float2 tau = make_float2(__fsub_ru(m.x, zmin.x), __fsub_ru(m.y, zmin.y));
      float2 den = make_float2(0.0f, 0.0f), psd = den;  // den, the sum of its rounded partial sums
#pragma unroll
      for (int k = 0; k < W; ++k) {
        pz[k] = softmax_exp_fast2(sub2_rn(pz[k], m));
        den = add2_rn(den, pz[k]);
        if (k > 0) psd = add2_ru(psd, den);
      }
      const float2 y = make_float2(__frcp_rn(den.x), __frcp_rn(den.y));
      // pooled sum, sum |terms|, sum |partial sums|
      float2 acc = make_float2(0.0f, 0.0f), aabs = acc, pss = acc;
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const uint32_t kw = lds_u32(reinterpret_cast<const uint32_t*>(&rb.kv[k][lane]) + c2);
        const float2 t = mul2_rn(mul2_rn(pz[k], y), make_float2(bf16_lo(kw), bf16_hi(kw)));
        acc = add2_rn(acc, t);
        aabs = add2_ru(aabs, abs2(t));
        if (k > 0) pss = add2_ru(pss, abs2(acc));
      }
      const float2 k2u = make_float2(B::k2u, B::k2u);
      // the weights' own and common relative bounds (Bounds), then sigma
      const float2 rown = fma2_rp(tau, make_float2(B::kC1u, B::kC1u), make_float2(B::kKown, B::kKown));
      const float2 rcom = fma2_rp(mul2_ru(psd, y), k2u, make_float2(B::kKcom, B::kKcom));
      const float2 sigma = mul2_ru(
          fma2_rp(add2_ru(rown, k2u), aabs, fma2_rp(rcom, abs2(acc), mul2_ru(k2u, pss))),
          make_float2(B::kWiden, B::kWiden));
      const float2 lo = sub2_rd(acc, sigma), hi = add2_ru(acc, sigma);
      ow[c2] = pack_bf16x2(lo.x, lo.y);
      const uint32_t diff = ow[c2] ^ pack_bf16x2(hi.x, hi.y);
      // in the range the bounds cover: tau <= kTMax, A finite (false for NaN)
      const bool ok0 = tau.x <= kTMax && aabs.x <= 1.2676506e30f;  // 2^100
      const bool ok1 = tau.y <= kTMax && aabs.y <= 1.2676506e30f;
      fbits |= (uint32_t)((diff & 0xFFFFu) != 0 || !ok0) << (2 * c2);
      fbits |= (uint32_t)((diff >> 16) != 0 || !ok1) << (2 * c2 + 1);
    }
    if (!col_ok) fbits = 0;
    // the warp's undecided columns, as lane * 4 + column, in rb.fail[0, n)
    int n = 0;
    if (__any_sync(0xffffffffu, fbits != 0)) {
#pragma unroll
      for (int i = 0; i < kCv; ++i) {
        const bool fail = (fbits >> i) & 1u;
        const uint32_t mc = __ballot_sync(0xffffffffu, fail);
        if (fail) rb.fail[n + __popc(mc & lt)] = (uint8_t)(lane * kCv + i);
        n += __popc(mc);
      }
    }
    if (col_ok) st_stream8(dst, make_uint2(ow[0], ow[1]));

    // queue the row's undecided columns; a full queue takes one exact pass
    for (int i = 0; i < n;) {
      const int take = min(n - i, kCap - pend);
      __syncwarp();
      for (int j = lane; j < take * W; j += 32) {
        const int en = j / W, k = j % W;
        const int e = rb.fail[i + en];
        const int lo = e >> 2, c = e & 3;  // owning lane and its column
        pq.sc[pend + en][k] = reinterpret_cast<const uint16_t*>(&rb.sc[k][lo])[c];
        pq.kv[pend + en][k] = reinterpret_cast<const uint16_t*>(&rb.kv[k][lo])[c];
      }
      if (lane < take) {
        const int e = rb.fail[i + lane];
        const int lo = e >> 2, c = e & 3;
        pq.tcol[pend + lane] = (uint16_t)((tx - lane + lo) * kCv + c);
        pq.off[pend + lane] = b * d + j0 + (lo - lane) * kCv + c;
      }
      pend += take;
      i += take;
      if (pend == kCap) {
        exact_pass(kCap);
        pend = 0;
      }
    }
  }
  if (pend > 0) exact_pass(pend);
}

template <int R, int COFF, int D>
cudaError_t launch_bitwise_d(const FwdParams& f, cudaStream_t stream) {
  constexpr int W = COFF * R;
  const int ncv = f.p.d / kCv;
  int tx = ncv <= 128 ? ncv : 128;
  tx = (tx + 31) / 32 * 32;  // whole warps in a row
  const int ty = kThreads / tx;
  const int tiles = (ncv + tx - 1) / tx;
  const size_t smem = sizeof(float) * W * tx * kCv +
                      (2 * sizeof(RowBuf<W>) + sizeof(Pending<W>)) * (size_t)(tx * ty / 32) +
                      seg_smem_bytes(f.p.nseq);
  auto kern = fwd_bitwise_kernel<R, COFF, D>;
  if (cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), 128 * 1024)) return e;
  const int occ = occupancy(reinterpret_cast<const void*>(kern), tx * ty, smem);
  const int64_t row_blocks = (f.p.C + ty - 1) / ty;
  int64_t gy = (int64_t)sm_count() * occ / tiles;
  if (gy < 1) gy = 1;
  if (gy > row_blocks) gy = row_blocks;
  if (gy > 65535) gy = 65535;
  return launch_dependent(kern, dim3(tiles, (unsigned)gy), dim3(tx, ty), smem, stream, f);
}

template <int R, int COFF>
cudaError_t launch_bitwise_rc(const FwdParams& f, cudaStream_t stream) {
  if (f.p.d == 512) return launch_bitwise_d<R, COFF, 512>(f, stream);
  if (f.p.d == 128) return launch_bitwise_d<R, COFF, 128>(f, stream);
  return launch_bitwise_d<R, COFF, 0>(f, stream);
}

}  // namespace

cudaError_t launch_fwd_bitwise(const FwdParams& f, cudaStream_t stream) {
  const Problem& p = f.p;
  if (p.C == 0) return cudaSuccess;
  switch (p.ratio * 4 + p.coff) {
    case 2 * 4 + 1: return launch_bitwise_rc<2, 1>(f, stream);
    case 2 * 4 + 2: return launch_bitwise_rc<2, 2>(f, stream);
    case 4 * 4 + 1: return launch_bitwise_rc<4, 1>(f, stream);
    case 4 * 4 + 2: return launch_bitwise_rc<4, 2>(f, stream);
    case 8 * 4 + 1: return launch_bitwise_rc<8, 1>(f, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csa
