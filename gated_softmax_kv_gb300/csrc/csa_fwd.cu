// Forward kernels of the CSA/HCA fused Compressor for sm_103a.
//
// cuDNN-frontend "CSA Fused Compressor", section "Semantics":
//   out[b, j] = sum_k kv[w(b,k), c(k,j)] * softmax_k(score[w(b,k), c(k,j)] + ape[k % ratio, c(k,j)])
// fp32 throughout, one final bf16 rounding (section "Numerics").
//
// The path is a streaming, HBM-bound pooling: each (token, column) element of
// kv and score is read exactly once (overlapping windows share tokens, never
// elements, because the two window halves use disjoint column ranges), so
// there is nothing for tensor cores or shared-memory reuse to win. Two
// kernel shapes:
//
//  * fwd_small (window W = coff*ratio <= 8): a thread owns one output row and
//    8 consecutive columns. It issues all 2W 16-byte loads of its window up
//    front (one coalesced 512-byte request per warp per slot), reads its APE
//    columns from a shared-memory slice staged once per CTA (persistent grid,
//    rows strided by the whole grid) and evaluates m = max z, e = exp(z - m),
//    den = sum e in slot order and out = (sum e * kv) / den: one division per
//    output instead of one per slot.
//
//  * fwd_long (W >= 16, e.g. ratio = 128; csa_fwd_long.cu): a thread owns 4
//    columns of one row and streams its window, or a chunk of it when few
//    rows would leave the GPU short of loads in flight, in batches of 8 slots
//    with an online softmax (running max, rescaled den and sum), prefetching
//    the next batch; chunk states merge in shared memory. Deterministic; the
//    rescaling reorders the sums, as the page's ratio = 128 kernels do.
//
// This file holds fwd_small, the dispatch over (ratio, coff) and the
// per-device helpers.
#include <cuda_runtime.h>
#include <stdint.h>

#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <utility>

#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

namespace {

constexpr int kThreads = 256;

// exp of the small-window forward, two lanes at a time. The forward has no
// bitwise target (the page's numerics give it "one bf16 rounding step on a
// tiny fraction of elements"), so it uses the single-rounding
// softmax_exp_fast: 5.6% faster at the headline than the compensated
// softmax_exp with the differing count unchanged within noise.
#ifndef CSA_FWD_EXP2
#define CSA_FWD_EXP2(x) softmax_exp_fast2(x)
#endif

// One output row's 8 columns from the window's kv / score vectors (masked
// slots already kv = 0, score = -inf) and the APE slice: logits z = score +
// ape, m = max z, e = exp(z - m), den = sum e in slot order, out = (sum e kv)
// / den, one bf16 rounding. The columns go in pairs through the two-lane fp32
// instructions (each lane rounded as the scalar operation).
template <int W>
__device__ __forceinline__ uint4 small_row_out(const uint4 (&kvv)[W], const uint4 (&scv)[W],
                                               const float* ape_s, int tile_cols) {
  float2 z[W][kVec / 2];
#pragma unroll
  for (int k = 0; k < W; ++k) {
    const float4 a0 = *reinterpret_cast<const float4*>(ape_s + k * tile_cols);
    const float4 a1 = *reinterpret_cast<const float4*>(ape_s + k * tile_cols + 4);
    z[k][0] = add2_rn(make_float2(bf16_lo(scv[k].x), bf16_hi(scv[k].x)), make_float2(a0.x, a0.y));
    z[k][1] = add2_rn(make_float2(bf16_lo(scv[k].y), bf16_hi(scv[k].y)), make_float2(a0.z, a0.w));
    z[k][2] = add2_rn(make_float2(bf16_lo(scv[k].z), bf16_hi(scv[k].z)), make_float2(a1.x, a1.y));
    z[k][3] = add2_rn(make_float2(bf16_lo(scv[k].w), bf16_hi(scv[k].w)), make_float2(a1.z, a1.w));
  }
  // m = max z, e = exp(z - m), den = sum e, out = (sum e * kv) / den
  uint32_t ow[4];
#pragma unroll
  for (int c2 = 0; c2 < 4; ++c2) {
    float m0 = z[0][c2].x, m1 = z[0][c2].y;
#pragma unroll
    for (int k = 1; k < W; ++k) {
      m0 = max_nan(m0, z[k][c2].x);
      m1 = max_nan(m1, z[k][c2].y);
    }
    const float2 m = make_float2(m0, m1);
    float2 den = make_float2(0.0f, 0.0f), acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < W; ++k) {
      const float2 e = CSA_FWD_EXP2(sub2_rn(z[k][c2], m));
      den = add2_rn(den, e);
      const uint32_t kw = c2 == 0 ? kvv[k].x : c2 == 1 ? kvv[k].y : c2 == 2 ? kvv[k].z : kvv[k].w;
      acc = fma2_rn(e, make_float2(bf16_lo(kw), bf16_hi(kw)), acc);
    }
    ow[c2] = pack_bf16x2(__fdiv_rn(acc.x, den.x), __fdiv_rn(acc.y, den.y));
  }
  return make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

// D > 0 fixes head_dim at compile time (slot offsets become immediates);
// D == 0 reads it from the problem.
// Windows of up to 4 slots fit three CTAs per SM (80 registers): 8-13% faster
// than two on the ratio-2 and ratio-4 coff-1 workloads (62766 ragged tokens at
// d 128, 8 x 4096 at d 512, 3 x 8192 at d 128, L2 flushed). W = 8 needs 128.
template <int R, int COFF, int D>
__global__ void __launch_bounds__(kThreads, (COFF * R <= 4 ? 3 : 2))
fwd_small_kernel(const FwdParams f) {
  grid_dependency_wait();
  allow_dependent_launch();
  constexpr int W = COFF * R;
  using S = Slot<R, COFF>;
  const Problem& p = f.p;
  const int d = D > 0 ? D : p.d;
  const int TX = blockDim.x, TY = blockDim.y;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int tid = ty * TX + tx, nthr = TX * TY;
  const int nvec = d / kVec;
  const int jv = blockIdx.x * TX + tx;
  const int64_t ld = (int64_t)COFF * d;
  const int j0 = jv * kVec;
  const int tile_cols = TX * kVec;
  // element offset of slot k from (row base token, column j0)
  auto koff = [&](int k) -> int64_t { return (S::tok(0, k)) * ld + S::half(k) * d; };

  // APE slice of this column tile, [W][tile_cols], read once per CTA, then
  // the segment arrays (seg_smem_bytes)
  extern __shared__ float sm[];
  for (int i = tid; i < W * tile_cols; i += nthr) {
    const int k = i / tile_cols;
    const int col = blockIdx.x * tile_cols + (i - k * tile_cols);
    sm[i] = col < d ? __ldg(p.ape + (int64_t)S::ape_row(k) * ld + S::half(k) * d + col) : 0.0f;
  }
  // then the segment arrays
  const SegMap sg = stage_segments(p.cu, p.cuc, p.nseq, reinterpret_cast<int32_t*>(sm + W * tile_cols),
                                   tid, nthr);
  __syncthreads();
  if (jv >= nvec) return;  // no barrier below
  const float* ape_s = sm + tx * kVec;

  const int64_t true_rows = sg.cuc[p.nseq];
  const int64_t stride = (int64_t)gridDim.y * TY;
  int hint = 0;
  // row b's window into kvv / scv (masked slots: kv = 0, score = -inf);
  // false, and nothing read, for a row that breaks the preconditions
  auto load_row = [&](int64_t b, uint4 (&kvv)[W], uint4 (&scv)[W]) -> bool {
    const RowInfo ri = row_info_from(sg.cu, sg.cuc, p.nseq, b, true_rows, R, hint);
    if (!row_in_bounds<R, COFF>(ri, p.T)) return false;
    const int64_t rowoff = ri.base * ld + j0;
#pragma unroll
    for (int k = 0; k < W; ++k) {
      if (S::masked(ri.first, k)) {
        kvv[k] = make_uint4(0u, 0u, 0u, 0u);
        scv[k] = make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
      } else {
        kvv[k] = ld_stream(p.kv + rowoff + koff(k));
        scv[k] = ld_stream(p.score + rowoff + koff(k));
      }
    }
    return true;
  };
  const uint4 nan4 = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
  // one row at a time (a next-row prefetch, which the small backward uses at
  // windows of up to 4 slots, measured slower here: 22.4 against 21.3 us at
  // ratio 2, coff 2, d 128, 62766 ragged tokens)
  for (int64_t b = (int64_t)blockIdx.y * TY + ty; b < p.C; b += stride) {
    uint4 kvv[W], scv[W];
    if (!load_row(b, kvv, scv)) {  // violated preconditions: NaN, no access
      st_stream(f.out + b * d + j0, nan4);
      continue;
    }
    st_stream(f.out + b * d + j0, small_row_out<W>(kvv, scv, ape_s, tile_cols));
  }
}

template <int R, int COFF, int D>
cudaError_t launch_small_d(const FwdParams& f, cudaStream_t stream) {
  constexpr int W = COFF * R;
  const int nvec = f.p.d / kVec;
  const int tx = nvec <= 128 ? nvec : 128;
  const int ty = kThreads / tx > 0 ? kThreads / tx : 1;
  const int tiles = (nvec + tx - 1) / tx;
  const size_t smem = sizeof(float) * W * tx * kVec + seg_smem_bytes(f.p.nseq);
  auto kern = fwd_small_kernel<R, COFF, D>;
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
cudaError_t launch_small(const FwdParams& f, cudaStream_t stream) {
  if (f.p.d == 512) return launch_small_d<R, COFF, 512>(f, stream);
  if (f.p.d == 128) return launch_small_d<R, COFF, 128>(f, stream);
  return launch_small_d<R, COFF, 0>(f, stream);
}

}  // namespace

bool supported(int ratio, int coff) {
  if (coff != 1 && coff != 2) return false;
  switch (ratio) {
    case 2: case 4: case 8: case 16: case 32: case 64: case 128: return true;
    default: return false;
  }
}

cudaError_t launch_fwd(const FwdParams& f, cudaStream_t stream) {
  if (f.p.C == 0) return cudaSuccess;
  if (f.p.exact) return launch_fwd_bitwise(f, stream);
  switch (f.p.ratio * 4 + f.p.coff) {
    case 2 * 4 + 1: return launch_small<2, 1>(f, stream);
    case 2 * 4 + 2: return launch_small<2, 2>(f, stream);
    case 4 * 4 + 1: return launch_small<4, 1>(f, stream);
    case 4 * 4 + 2: return launch_small<4, 2>(f, stream);
    case 8 * 4 + 1: return launch_small<8, 1>(f, stream);
    default: return launch_fwd_long(f, stream);  // windows of 16 slots and more
  }
}

int occupancy(const void* kernel, int threads, size_t smem) {
  // cached per (kernel, device, block size, shared memory): the grids of a
  // call depend on it and the query costs host time on every call otherwise
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, size_t>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  const auto key = std::make_tuple(kernel, dev, threads, smem);
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, threads, smem) != cudaSuccess ||
      blocks < 1)
    return 1;  // not cached: a failed query is retried next time
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = blocks;
  return blocks;
}

cudaError_t allow_dynamic_smem(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  if (cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))
    return e;
  done.insert({kernel, dev});
  return cudaSuccess;
}

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace csa
