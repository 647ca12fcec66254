// Bitwise backward of the CSA/HCA fused Compressor for windows of W <= 8 slots
// (sm_103a).
//
// cuDNN-frontend "CSA Fused Compressor", section "Numerics": for ratios 2 and 4
// the page's backward gives dKV / dScore bit-identical to the fp32 eager
// reference. This kernel gives the bits of the fp32 eager-order reference of
// this library (correctly rounded exp, e / den with IEEE division, slot-order
// sums from +0, every product and sum rounded separately, one bf16 rounding)
// while keeping the streaming kernel's arithmetic for almost every element.
//
// Per (row, column) the kernel
//  1. runs the fast path of the default backward (exp(x) = ex2.approx(RN(x
//     log2 e)), p = e RN(1/den), S = sum RN(dp p) in slot order);
//  2. encloses the reference's fp32 results from it. With t_k = z_k - m the
//     reference's exp argument (the fast path computes the same z, m, t), the
//     fast exp is within eps(t) = (kExpC1 |t| + kExpC0) 2^-24 relative of the
//     correctly rounded exp for t in [-kTMax, 0] (checked on every fp32 t of
//     that range by the GPU tests). A sequential sum differs from the exact
//     sum of its terms by at most 2^-24 times the sum of its rounded partial
//     sums, on either side. From these, with tau >= max |t_k| over the
//     window's valid slots:
//       p_ref = p (1 + delta_k)(1 + Delta), |delta_k| <= rho_own, |Delta| <= rho_com,
//       rho_own = (kExpC1 tau + kExpC0 + 2.5) 2^-24,
//       rho_com = (kExpC0 + kExpC1 (W - 1) / e + 1.5) 2^-24 + 2^-23 P_den / den:
//     the slot's own exp, product and quotient roundings; and, common to the
//     column, the exps' weighted contribution to den (at most kExpC0 +
//     kExpC1 (W - 1) / e, since t e^t >= -1/e and den >= 1), both sides' den
//     rounding (P_den = the sum of den's partial sums) and the reciprocal
//     (each bound also covers the inversion of the ratio); so p_ref lies in
//     p [1 - rho, 1 + rho], rho = rho_own + rho_com; and, since the common
//     factor scales the whole sum,
//       S_ref in [S - sigma, S + sigma],
//       sigma = (rho_own + 2^-23) A + rho_com |S| + 2^-23 P_S,
//     with A = sum |RN(dp p)| and P_S the sum of |S's partial sums|. Each
//     enclosure is then pushed through the
//     reference's own monotone steps with directed rounding:
//       dkv_ref = RN(g p_ref)        in [RN(g_a p), RN(g_b p)],
//         g_a = RD(g - rho |g|), g_b = RU(g + rho |g|), each given the sign
//         of g (so that g = +0 or -0 gives its own zero at both ends);
//       diff_ref = RN(dp - S_ref)    in [RN(dp - S_hi), RN(dp - S_lo)] = [dl, dh],
//       dz_ref = RN(p_ref diff_ref)  in [RN(p RD(dl - rho |dl|)), RN(p RU(dh + rho |dh|))],
//     using that RN is monotone and p > 0 (signed zeros included: an
//     enclosure whose two ends differ in sign fails the test below);
//  3. accepts the fast path's bits for the column when every enclosure's two
//     ends round to the same bf16 bits (then so does the reference's value,
//     which lies between them) and the column is in the range the bounds
//     cover (tau <= kTMax, so every weight is a normal number, and A finite);
//  4. otherwise recomputes the column exactly after the fast stores of the
//     row, from the row's inputs in shared memory (rows arrive there by
//     cp.async one row ahead of their computation): the warp's failing
//     columns are taken W / 2 lanes per column (two window slots a lane:
//     correctly rounded exp, correctly rounded division, the reference's
//     slot-order den and S summed by every lane of the column from gathered
//     values), eight columns per pass at W = 8, and the exact bf16 values
//     overwrite the fast ones while those lines are still in L2. Windows of
//     up to 4 slots (16- or 32-column passes, about 2 failing columns a
//     row) copy their failing columns into a per-warp queue instead, and a
//     full queue, or at the end what is left in it, takes one pass.
// dape sums the midpoints of the dz enclosures (deterministically, in the
// two fixed-order levels of the default backward); zero writes and row
// groups are those of the default small-window backward.
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa_bwd_common.cuh"
#include "csa_device.cuh"
#include "csa_bitwise.cuh"
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
bwd_bitwise_kernel(const BwdParams bp) {
  grid_dependency_wait();
  allow_dependent_launch();
  constexpr int W = COFF * R;
  constexpr int L = W / 2;   // lanes per column in the exact pass
  constexpr int P = 32 / L;  // columns per exact pass
  using S = Slot<R, COFF>;
  using B = Bounds<W>;
  const Problem& p = bp.p;
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

  // [W][tile_cols] APE slice (later the dape combine buffer), then two row
  // buffers per warp (the current row and the next one, in flight)
  extern __shared__ float sm[];
  __shared__ float tab[2 * kExpTableSize];
  exp_cr_table(tab);
  for (int i = tid; i < W * tile_cols; i += nthr) {
    const int k = i / tile_cols;
    const int col = blockIdx.x * tile_cols + (i - k * tile_cols);
    sm[i] = col < d ? __ldg(p.ape + (int64_t)S::ape_row(k) * ld + S::half(k) * d + col) : 0.0f;
  }
  __syncthreads();
  const float* ape_s = sm + tx * kCv;
  RowBuf<W>* const rb0 = reinterpret_cast<RowBuf<W>*>(sm + W * tile_cols);
  RowBuf<W>* rbs = rb0 + 2 * (tid >> 5);
  // windows of up to 4 slots queue their undecided columns (few per row for
  // passes of 16 or 32 columns); W = 8 runs one pass per row with failures
  constexpr bool kQueue = W <= 4;
  Pending<W>& pq = reinterpret_cast<Pending<W>*>(rb0 + 2 * (nthr >> 5))[tid >> 5];
  constexpr int kCap = Pending<W>::kCap;
  static_assert(kCap == P, "a pass takes the whole queue");

  float2 dacc[W][kCv / 2];  // sums of dz_lo + dz_hi (twice dz), per column pair
#pragma unroll
  for (int k = 0; k < W; ++k)
#pragma unroll
    for (int c2 = 0; c2 < kCv / 2; ++c2) dacc[k][c2] = make_float2(0.0f, 0.0f);

  const uint2 zero2 = make_uint2(0u, 0u);
  // the segment arrays stay in global memory here: a row looks up the row
  // after it a full row ahead of its use, and the registers of a shared
  // copy's pointers are what this kernel lacks
  const int64_t true_rows = __ldg(p.cuc + p.nseq);
  const int64_t stride = (int64_t)gridDim.y * TY;
  const uint32_t lt = (1u << lane) - 1u;
  int hint = 0;

  // The window of row `row` into `buf`: asynchronous copies of kv, score and
  // grad_out (constants for masked slots and lanes without columns); rows
  // that read nothing (out of bounds, past capacity) copy nothing.
  auto fetch = [&](int64_t row, const RowInfo& info, RowBuf<W>& buf) {
    if (!row_in_bounds<R, COFF>(info, p.T) || row >= p.C) return;
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
    if (col_ok) cp_async8(&buf.g[lane], bp.grad_out + row * d + j0);
    else buf.g[lane] = zero2;
  };

  // The exact pass over the first cnt queued columns: as the per-row pass
  // below, reading the columns from the queue.
  auto queued_pass = [&](int cnt) {
    const int q = lane / L, l = lane % L, gbase = lane & ~(L - 1);
    const int k0 = 2 * l, k1 = 2 * l + 1;
    __syncwarp();
    const bool act = q < cnt;
    const int qe = act ? q : 0;
    const uint32_t sw = lds_u32(&pq.sc[qe][k0]);  // slots k0 and k1
    const uint32_t kw = lds_u32(&pq.kv[qe][k0]);
    const uint16_t gh = pq.g[qe];
    const float g = __uint_as_float((uint32_t)gh << 16);
    const int tcol = pq.tcol[qe];
    const bool first = pq.first[qe];
    uint16_t s0, s1, v0, v1;
    split_bf16x2(sw, s0, s1);
    split_bf16x2(kw, v0, v1);
    const float2 z = make_float2(add_bf16_f32(s0, sm[k0 * tile_cols + tcol]),
                                 add_bf16_f32(s1, sm[k1 * tile_cols + tcol]));
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
    const float dp0 = mul_bf16(gh, v0), dp1 = mul_bf16(gh, v1);  // RN(g kv), exact
    const float t0 = __fmul_rn(dp0, pw.x), t1 = __fmul_rn(dp1, pw.y);
    float sfin = 0.0f;
#pragma unroll
    for (int k = 0; k < W; ++k)
      sfin = __fadd_rn(sfin, __shfl_sync(0xffffffffu, (k & 1) ? t1 : t0, gbase + k / 2));
    if (act) {
      uint16_t* dk = bp.dkv + pq.off[qe];
      uint16_t* dz = bp.dscore + pq.off[qe];
      if (!S::masked(first, k0)) {
        st_u16(dk + koff(k0), bf16_bits_rn(__fmul_rn(g, pw.x)));
        st_u16(dz + koff(k0), bf16_bits_rn(__fmul_rn(pw.x, __fsub_rn(dp0, sfin))));
      }
      if (!S::masked(first, k1)) {
        st_u16(dk + koff(k1), bf16_bits_rn(__fmul_rn(g, pw.y)));
        st_u16(dz + koff(k1), bf16_bits_rn(__fmul_rn(pw.y, __fsub_rn(dp1, sfin))));
      }
    }
    __syncwarp();
  };
  int pend = 0;  // queued columns

  // every lane of a warp runs every row of its warp (the exact pass is warp-wide)
  int64_t b = (int64_t)blockIdx.y * TY + ty;
  if (b < true_rows) fetch(b, row_info_from<true>(p.cu, p.cuc, p.nseq, b, true_rows, R, hint), rbs[0]);
  cp_async_commit();
  for (int it = 0; b < true_rows; ++it, b += stride) {
    // the row's map (rows are visited in increasing order, so the segment
    // hint makes this one cached load), then the next row into the other
    // buffer, last read by the previous row
    const RowInfo cur = row_info_from<true>(p.cu, p.cuc, p.nseq, b, true_rows, R, hint);
    __syncwarp();
    if (b + stride < true_rows)
      fetch(b + stride, row_info_from<true>(p.cu, p.cuc, p.nseq, b + stride, true_rows, R, hint),
            rbs[(it + 1) & 1]);
    cp_async_commit();
    cp_async_wait<1>();  // this row's copies have landed ...
    __syncwarp();        // ... for every lane of the warp
    RowBuf<W>& rb = rbs[it & 1];
    if (!row_in_bounds<R, COFF>(cur, p.T)) continue;  // violated preconditions: skip
    const int64_t rowoff = cur.base * ld + j0;
    uint16_t* dkv_row = bp.dkv + rowoff;
    uint16_t* dsc_row = bp.dscore + rowoff;
    if (b < p.C) {
      // per column pair (the two lanes of f32x2 values): z = score + ape,
      // then in place e, then p; then the pair's bf16 outputs
      float2 pz[W][2];
      int n = 0;  // failing columns of the row so far
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        // the pair's kv and score words, from the row buffer
        uint32_t kw[W];
#pragma unroll
        for (int k = 0; k < W; ++k) {
          const float2 a = *reinterpret_cast<const float2*>(ape_s + k * tile_cols + 2 * c2);
          const uint32_t w = lds_u32(reinterpret_cast<const uint32_t*>(&rb.sc[k][lane]) + c2);
          kw[k] = lds_u32(reinterpret_cast<const uint32_t*>(&rb.kv[k][lane]) + c2);
          uint16_t s0, s1;
          split_bf16x2(w, s0, s1);
          pz[k][c2] = make_float2(add_bf16_f32(s0, a.x), add_bf16_f32(s1, a.y));
        }
        const uint32_t gw = lds_u32(reinterpret_cast<const uint32_t*>(&rb.g[lane]) + c2);
        uint16_t g0, g1;
        split_bf16x2(gw, g0, g1);
        auto zx = [&](int k) { return pz[k][c2].x; };
        auto zy = [&](int k) { return pz[k][c2].y; };
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
          pz[k][c2] = softmax_exp_fast2(sub2_rn(pz[k][c2], m));
          den = add2_rn(den, pz[k][c2]);
          if (k > 0) psd = add2_ru(psd, den);
        }
        const float2 y = make_float2(__frcp_rn(den.x), __frcp_rn(den.y));
#pragma unroll
        for (int k = 0; k < W; ++k) pz[k][c2] = mul2_rn(pz[k][c2], y);
        const float2 g2 = make_float2(bf16_lo(gw), bf16_hi(gw));
        // S, sum |terms|, sum |partial sums|
        float2 acc = make_float2(0.0f, 0.0f), aabs = acc, pss = acc;
#pragma unroll
        for (int k = 0; k < W; ++k) {
          uint16_t v0, v1;
          split_bf16x2(kw[k], v0, v1);
          const float2 dp = make_float2(mul_bf16(g0, v0), mul_bf16(g1, v1));  // RN(g kv)
          const float2 t = mul2_rn(dp, pz[k][c2]);
          acc = add2_rn(acc, t);
          aabs = add2_ru(aabs, abs2(t));
          if (k > 0) pss = add2_ru(pss, abs2(acc));
        }
        const float2 k2u = make_float2(B::k2u, B::k2u);
        // the weights' own and common relative bounds (Bounds): rho = their
        // sum for dkv and dz, the common one against |S| in sigma
        const float2 rown = fma2_rp(tau, make_float2(B::kC1u, B::kC1u), make_float2(B::kKown, B::kKown));
        const float2 rcom = fma2_rp(mul2_ru(psd, y), k2u, make_float2(B::kKcom, B::kKcom));
        const float2 rho2 = add2_ru(rown, rcom);
        const float2 nrho2 = make_float2(-rho2.x, -rho2.y);
        const float2 sigma = mul2_ru(
            fma2_rp(add2_ru(rown, k2u), aabs, fma2_rp(rcom, abs2(acc), mul2_ru(k2u, pss))),
            make_float2(B::kWiden, B::kWiden));
        const float2 slo2 = sub2_rd(acc, sigma), shi2 = add2_ru(acc, sigma);
        // g -/+ rho |g| rounded outwards, with the sign of g: the directed
        // roundings give -0 / +0 at g = +0 / -0, and g p_ref has g's sign
        const float2 ga = fma2_rm(abs2(g2), nrho2, g2), gb = fma2_rp(abs2(g2), rho2, g2);
        const float2 ga2 = make_float2(copysignf(ga.x, g2.x), copysignf(ga.y, g2.y));
        const float2 gb2 = make_float2(copysignf(gb.x, g2.x), copysignf(gb.y, g2.y));
        // in the range the bounds cover: tau <= kTMax, A finite (false for NaN)
        const bool ok0 = tau.x <= kTMax && aabs.x <= 1.2676506e30f;  // 2^100
        const bool ok1 = tau.y <= kTMax && aabs.y <= 1.2676506e30f;
        uint32_t diff = 0;
#pragma unroll
        for (int k = 0; k < W; ++k) {
          const float2 pk = pz[k][c2];
          // the reference's dp = RN(g kv) as bf16 FMAs with a -0 addend: no
          // later step can fuse them, and dl / dh need that dp
          const uint32_t kwk = lds_u32(reinterpret_cast<const uint32_t*>(&rb.kv[k][lane]) + c2);
          uint16_t v0, v1;
          split_bf16x2(kwk, v0, v1);
          const float2 dp = make_float2(mul_bf16(g0, v0), mul_bf16(g1, v1));
          const float2 dl = sub2_rn(dp, shi2), dh = sub2_rn(dp, slo2);
          const float2 zl = mul2_rn(pk, fma2_rm(abs2(dl), nrho2, dl));
          const float2 zh = mul2_rn(pk, fma2_rp(abs2(dh), rho2, dh));
          const float2 dka = mul2_rn(ga2, pk), dkb = mul2_rn(gb2, pk);
          const uint32_t wka = pack_bf16x2(dka.x, dka.y);
          const uint32_t wzl = pack_bf16x2(zl.x, zl.y);
          if (!S::masked(cur.first, k))
            diff |= (wka ^ pack_bf16x2(dkb.x, dkb.y)) | (wzl ^ pack_bf16x2(zh.x, zh.y));
          dacc[k][c2] = add2_rn(dacc[k][c2], add2_rn(zl, zh));
          // dkv and dscore words of columns 2 c2 and 2 c2 + 1, stored now: holding
          // them for 8-byte stores after the second pair spilled
          if (col_ok && !S::masked(cur.first, k)) {
            st_u32_na(dkv_row + koff(k) + 2 * c2, wka);
            st_u32_na(dsc_row + koff(k) + 2 * c2, wzl);
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const bool fail = col_ok && (((h ? diff >> 16 : diff & 0xFFFFu) != 0) || !(h ? ok1 : ok0));
          const uint32_t mc = __ballot_sync(0xffffffffu, fail);
          if (fail) rb.fail[n + __popc(mc & lt)] = (uint8_t)(lane * kCv + 2 * c2 + h);
          n += __popc(mc);
        }
      }

      if constexpr (kQueue) {
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
            pq.g[pend + lane] = reinterpret_cast<const uint16_t*>(&rb.g[lo])[c];
            pq.tcol[pend + lane] = (uint16_t)((tx - lane + lo) * kCv + c);
            pq.first[pend + lane] = cur.first;
            pq.off[pend + lane] = rowoff + (lo - lane) * kCv + c;
          }
          pend += take;
          i += take;
          if (pend == kCap) {
            queued_pass(kCap);
            pend = 0;
          }
        }
      } else if (n > 0) {
        // ---- exact pass over the warp's failing columns of this row ----
        const int q = lane / L, l = lane % L, gbase = lane & ~(L - 1);
        const int k0 = 2 * l, k1 = 2 * l + 1;
        const bool m0 = S::masked(cur.first, k0), m1 = S::masked(cur.first, k1);
        __syncwarp();
        for (int base = 0; base < n; base += P) {
          const bool act = base + q < n;
          const int e = rb.fail[act ? base + q : base];
          const int lo = e >> 2, c = e & 3;  // owning lane and its column
          const uint16_t* kv16 = reinterpret_cast<const uint16_t*>(&rb.kv[0][lo]) + c;
          const uint16_t* sc16 = reinterpret_cast<const uint16_t*>(&rb.sc[0][lo]) + c;
          constexpr int kStride = 32 * 4;  // 16-bit units from one slot's words to the next
          // masked slots hold score -inf and kv 0 in the row buffer, as copied in
          const uint16_t s0 = sc16[k0 * kStride], s1 = sc16[k1 * kStride];
          const uint16_t v0 = kv16[k0 * kStride], v1 = kv16[k1 * kStride];
          const uint16_t gh = reinterpret_cast<const uint16_t*>(&rb.g[lo])[c];
          const float g = __uint_as_float((uint32_t)gh << 16);
          const int tcol = (tx - lane + lo) * kCv + c;
          const float2 z = make_float2(add_bf16_f32(s0, sm[k0 * tile_cols + tcol]),
                                       add_bf16_f32(s1, sm[k1 * tile_cols + tcol]));
          float mx = max_nan(z.x, z.y);
#pragma unroll
          for (int o = 1; o < L; o <<= 1) mx = max_nan(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          const float2 ex = exp_cr2(sub2_rn(z, make_float2(mx, mx)), tab);
          // den and S in slot order: every lane of the column's group gathers
          // the W values (independent shuffles) and sums them itself
          float den = 0.0f;
#pragma unroll
          for (int k = 0; k < W; ++k)
            den = __fadd_rn(den, __shfl_sync(0xffffffffu, (k & 1) ? ex.y : ex.x, gbase + k / 2));
          const float yd = __frcp_rn(den);
          const float2 pw = div2_cr(ex, make_float2(den, den), make_float2(-den, -den),
                                    make_float2(yd, yd));
          const float dp0 = mul_bf16(gh, v0), dp1 = mul_bf16(gh, v1);  // RN(g kv), exact
          const float t0 = __fmul_rn(dp0, pw.x), t1 = __fmul_rn(dp1, pw.y);
          float sfin = 0.0f;
#pragma unroll
          for (int k = 0; k < W; ++k)
            sfin = __fadd_rn(sfin, __shfl_sync(0xffffffffu, (k & 1) ? t1 : t0, gbase + k / 2));
          if (act) {
            const int64_t off = rowoff + (lo - lane) * kCv + c;
            uint16_t* dk = bp.dkv + off;
            uint16_t* dz = bp.dscore + off;
            if (!m0) {
              st_u16(dk + koff(k0), bf16_bits_rn(__fmul_rn(g, pw.x)));
              st_u16(dz + koff(k0), bf16_bits_rn(__fmul_rn(pw.x, __fsub_rn(dp0, sfin))));
            }
            if (!m1) {
              st_u16(dk + koff(k1), bf16_bits_rn(__fmul_rn(g, pw.y)));
              st_u16(dz + koff(k1), bf16_bits_rn(__fmul_rn(pw.y, __fsub_rn(dp1, sfin))));
            }
          }
        }
      }
    } else if (col_ok) {
      // a row past capacity has no output slot: zero gradient at its positions
#pragma unroll
      for (int k = 0; k < W; ++k) {
        if (S::masked(cur.first, k)) continue;
        st_stream8(dkv_row + koff(k), zero2);
        st_stream8(dsc_row + koff(k), zero2);
      }
    }
    if (cur.last && col_ok) {
      // the segment's last row owns its block's unread first-half columns ...
      if (COFF == 2) {
#pragma unroll
        for (int t = 0; t < R; ++t) {
          st_stream8(dkv_row + t * ld, zero2);
          st_stream8(dsc_row + t * ld, zero2);
        }
      }
      // ... and the segment's tail tokens (seqlen % ratio of them)
      const int64_t tail_end = cur.seg_end < p.T ? cur.seg_end : p.T;
      for (int64_t tok = cur.base + R; tok < tail_end; ++tok) {
#pragma unroll
        for (int h = 0; h < COFF; ++h) {
          const int64_t off = tok * ld + h * d + j0;
          st_stream8(bp.dkv + off, zero2);
          st_stream8(bp.dscore + off, zero2);
        }
      }
    }
  }
  if constexpr (kQueue) {
    if (pend > 0) queued_pass(pend);
  }
  cp_async_wait<0>();

  zero_orphans(bp, R);

  // combine the TY thread rows in ascending order, then write this CTA's
  // slice of the partial of row group blockIdx.y (halving the sums of the
  // two enclosure ends: exact)
  __syncthreads();
  for (int t = 0; t < TY; ++t) {
    if (ty == t && col_ok) {
#pragma unroll
      for (int k = 0; k < W; ++k)
#pragma unroll
        for (int c2 = 0; c2 < kCv / 2; ++c2) {
          float2* s = reinterpret_cast<float2*>(sm + k * tile_cols + tx * kCv + 2 * c2);
          *s = t == 0 ? dacc[k][c2] : add2_rn(*s, dacc[k][c2]);
        }
    }
    __syncthreads();
  }
  float* part = bp.partial + (int64_t)blockIdx.y * (R * ld);
  for (int i = tid; i < W * tile_cols; i += nthr) {
    const int k = i / tile_cols;
    const int col = blockIdx.x * tile_cols + (i - k * tile_cols);
    if (col < d) part[(int64_t)S::ape_row(k) * ld + S::half(k) * d + col] = 0.5f * sm[i];
  }
}

template <int R, int COFF, int D>
cudaError_t plan_bitwise_d(const Problem& p, BwdShape* s) {
  constexpr int W = COFF * R;
  const int ncv = p.d / kCv;
  int tx = ncv <= 128 ? ncv : 128;
  tx = (tx + 31) / 32 * 32;  // whole warps in a row
  const int ty = kThreads / tx;
  const int tiles = (ncv + tx - 1) / tx;
  // the queue of undecided columns at windows of up to 4 slots (the kernel's kQueue)
  const size_t smem = sizeof(float) * W * tx * kCv +
                      (2 * sizeof(RowBuf<W>) + (W <= 4 ? sizeof(Pending<W>) : 0)) * (size_t)(tx * ty / 32);
  auto kern = bwd_bitwise_kernel<R, COFF, D>;
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
cudaError_t plan_bitwise_rc(const Problem& p, BwdShape* s) {
  if (p.d == 512) return plan_bitwise_d<R, COFF, 512>(p, s);
  if (p.d == 128) return plan_bitwise_d<R, COFF, 128>(p, s);
  return plan_bitwise_d<R, COFF, 0>(p, s);
}

template <int R, int COFF>
cudaError_t run_bitwise_rc(const BwdParams& b, const BwdShape& s, cudaStream_t stream) {
  auto kern = b.p.d == 512 ? bwd_bitwise_kernel<R, COFF, 512>
             : b.p.d == 128 ? bwd_bitwise_kernel<R, COFF, 128> : bwd_bitwise_kernel<R, COFF, 0>;
  return launch_dependent(kern, s.grid, s.block, s.smem, stream, b);
}

#define CSA_BITWISE_DISPATCH(FN, ...)               \
  switch (p.ratio * 4 + p.coff) {                   \
    case 2 * 4 + 1: return FN<2, 1>(__VA_ARGS__);   \
    case 2 * 4 + 2: return FN<2, 2>(__VA_ARGS__);   \
    case 4 * 4 + 1: return FN<4, 1>(__VA_ARGS__);   \
    case 4 * 4 + 2: return FN<4, 2>(__VA_ARGS__);   \
    case 8 * 4 + 1: return FN<8, 1>(__VA_ARGS__);   \
    default: return cudaErrorInvalidValue;          \
  }

}  // namespace

cudaError_t plan_bwd_bitwise(const Problem& p, BwdShape* shape) {
  CSA_BITWISE_DISPATCH(plan_bitwise_rc, p, shape)
}

cudaError_t launch_bwd_bitwise(const BwdParams& b, const BwdShape& shape, cudaStream_t stream) {
  const Problem& p = b.p;
  CSA_BITWISE_DISPATCH(run_bitwise_rc, b, shape, stream)
}

}  // namespace csa
