/*
 * csa_compress.h -- C ABI of the GB300 (sm_103a) CSA/HCA fused Compressor.
 *
 * The operation (cuDNN-frontend "CSA Fused Compressor", section "Semantics"):
 * for every THD segment s (tokens cu_seqlens[s] .. cu_seqlens[s+1]) and every
 * output block b of `ratio` tokens,
 *
 *   out[b, j] = sum_k kv[w(b,k), c(k,j)] * softmax_k(score[w(b,k), c(k,j)]
 *                                                     + ape[k % ratio, c(k,j)])
 *
 * with the overlapping window (coff == 2, 2*ratio slots: k < ratio reads the
 * previous block's token on first-half column j with APE row k, masked on a
 * segment's first block; k >= ratio reads the own block's token on
 * second-half column head_dim + j with APE row k - ratio) or the own-block
 * window (coff == 1, ratio slots, column j, APE row k, never masked). A
 * segment's seqlen % ratio tail tokens are never read. Output rows
 * b >= cu_seqlens_comp[num_seqs] up to `capacity` (static CUDA-graph
 * capacity) are computed as a first block whose own tokens are 0..ratio-1;
 * the backward ignores grad_out on those rows. Arithmetic is fp32 with one
 * final bf16 rounding (section "Numerics").
 *
 * Layouts (row-major, contiguous, all on the current CUDA device):
 *   kv, score     bf16 [total_tokens, coff*head_dim]; for coff == 2 columns
 *                 [0, head_dim) are the first half, [head_dim, 2*head_dim) the second
 *   ape           fp32 [ratio, coff*head_dim]
 *   cu_seqlens    int32 [num_seqs + 1]   token prefix sums, cu_seqlens[0] == 0
 *   cu_seqlens_comp int32 [num_seqs + 1] prefix sums of floor(seqlen / ratio)
 *   out, grad_out bf16 [capacity, head_dim]
 *   dkv, dscore   bf16 [total_tokens, coff*head_dim]
 *   dape          fp32 [ratio, coff*head_dim]
 *
 * Ownership: every pointer is caller-owned device memory; nothing is retained
 * after a call returns. Calls are asynchronous on `stream` and never
 * synchronise the host. The segment arrays are read on the device only.
 *
 * Supported envelope (checked on the host before any launch, otherwise an
 * error is returned and nothing is launched or written):
 *   ratio in {2, 4, 8, 16, 32, 64, 128}, coff in {1, 2}, head_dim % 8 == 0,
 *   head_dim >= 8, num_seqs >= 1, total_tokens >= 0, capacity >= 0,
 *   total_tokens * coff * head_dim < 2^31 and capacity * head_dim < 2^31
 *   (section "Support surface", int32 flat offsets), capacity > 0 requires
 *   total_tokens >= ratio, 16-byte aligned kv/score/ape/out/grad_out/dkv/
 *   dscore/dape and 4-byte aligned segment arrays, no null pointer.
 *
 * Device-side preconditions (not checked by the compute calls: checking them
 * would need a host synchronisation; csa_check_segments below checks them on
 * request): cu_seqlens and cu_seqlens_comp start at 0 and do not
 * decrease, cu_seqlens[num_seqs] <= total_tokens,
 * cu_seqlens_comp[s+1] - cu_seqlens_comp[s] == floor(seqlen_s / ratio).
 * When they do not hold the kernels still stay inside the buffers described
 * above, but the contents of the outputs are unspecified. When
 * cu_seqlens_comp[num_seqs] > capacity the rows beyond capacity have no
 * output slot: the backward treats them as rows with zero gradient.
 */
#ifndef CSA_COMPRESS_H
#define CSA_COMPRESS_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum csa_status {
  CSA_OK = 0,
  CSA_ERR_NULL = 1,        /* a required pointer is null                          */
  CSA_ERR_ALIGN = 2,       /* a base pointer is not aligned as required           */
  CSA_ERR_UNSUPPORTED = 3, /* ratio / coff / head_dim outside the envelope        */
  CSA_ERR_RANGE = 4,       /* a size is negative or overflows int32 flat offsets  */
  CSA_ERR_CUDA = 5,        /* a CUDA runtime call failed (see csa_last_cuda_error) */
  CSA_ERR_SCRATCH = 6      /* csa_compress_bwd_noalloc: the call needs more dape scratch
                              than the library's fixed device buffer holds            */
} csa_status_t;

/*
 * Forward. Writes out[b, :] for every b in [0, capacity) (padding rows
 * included). capacity == 0 launches nothing. One kernel launch.
 */
csa_status_t csa_compress_fwd(const void* kv, const void* score, const float* ape,
                              const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                              int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                              int32_t ratio, int32_t coff, int32_t head_dim,
                              void* out, cudaStream_t stream);

/*
 * Backward (cuDNN-frontend "CSA Fused Compressor", sections "Semantics" and
 * "Class API"). Recomputes the softmax weights and writes:
 *   dkv, dscore -- EVERY element of [total_tokens, coff*head_dim]: the gradient
 *                  at positions a non-padding row reads, exact +0 at every
 *                  position no such row reads (segment tails, the first-half
 *                  columns of a segment's last block, segments shorter than
 *                  ratio, tokens >= cu_seqlens[num_seqs]). They may be
 *                  uninitialised on entry.
 *   dape        -- OVERWRITTEN (not accumulated) with the sum over non-padding
 *                  rows of every window slot's fp32 logit gradient, reduced in
 *                  a fixed order (per-block fp32 partials, then an ordered
 *                  final sum): bitwise run-to-run deterministic, no atomics;
 *                  the row grouping, like every other choice that orders
 *                  the arithmetic, depends on the problem only, never on the
 *                  device's SM count.
 * grad_out rows >= cu_seqlens_comp[num_seqs] are never read.
 * Two kernel launches. The dape partials live in a stream-ordered workspace
 * taken from a library-owned CUDA memory pool on `stream` (released on the
 * stream after use, kept cached by the pool). The pool belongs to the CUDA
 * context current at the call; after a device reset the next call makes a new
 * one.
 */
csa_status_t csa_compress_bwd(const void* kv, const void* score, const float* ape,
                              const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                              int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                              int32_t ratio, int32_t coff, int32_t head_dim,
                              const void* grad_out, void* dkv, void* dscore, float* dape,
                              cudaStream_t stream);

/*
 * Backward that allocates no device memory. This entry point has no
 * counterpart in the paper; it exists for callers that cannot allocate device
 * memory while they run the backward -- for example a process that hands all
 * of its device memory to its own allocator at start-up, or a time-critical
 * loop that must not enter the CUDA allocator (csa_compress_bwd takes its dape
 * workspace from a stream-ordered memory pool, which can grow on first use).
 *
 * Same arguments, outputs and numerics as csa_compress_bwd (same kernels,
 * same launch shape, so the results are bitwise identical). The dape partials
 * live in one fixed array of CSA_NOALLOC_SCRATCH_FLOATS floats (16 MiB) that
 * the library reserves statically on every GPU that loads it, for the life of
 * the process. A call whose partials do not fit returns CSA_ERR_SCRATCH before
 * launching anything. The need is ratio * coff * head_dim floats per row
 * group; the row groups number at most 152 x resident blocks per SM / column
 * tiles, so the product does not grow with head_dim, and it depends on the
 * problem alone (the row grouping never depends on the device): 1.2 Mi
 * floats at the 256k-token ratio-4 headline, 2.4 Mi at ratio 128 (coff 1,
 * head_dim 512). Only a single group larger than the buffer exhausts it:
 * ratio 128, coff 2, head_dim 16384 needs exactly 4 Mi (accepted), head_dim
 * 16392 is refused.
 *
 * The first call in a CUDA context of a device looks up that array's device
 * address (with the caller's device current) and keeps it for the context;
 * make that first call before any stream capture. After the context is
 * destroyed and created again (cudaDeviceReset), the next call looks the
 * address up afresh; the array's contents do not survive the reset. All calls
 * share the one array and leave their partials in it: calls whose kernels
 * overlap on the GPU (different streams, or several host threads) race on it
 * and must be serialised by the caller. Nothing in the array needs clearing
 * between calls: each call overwrites every partial it reads.
 */
#define CSA_NOALLOC_SCRATCH_FLOATS (4 * 1024 * 1024)
csa_status_t csa_compress_bwd_noalloc(const void* kv, const void* score, const float* ape,
                                      const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                                      int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                                      int32_t ratio, int32_t coff, int32_t head_dim,
                                      const void* grad_out, void* dkv, void* dscore, float* dape,
                                      cudaStream_t stream);

/*
 * Exact mode (cuDNN-frontend "CSA Fused Compressor", section "Numerics":
 * bitwise agreement with an fp32 eager reference is the aim for ratios 2 and
 * 4). Same arguments, layouts, outputs and ownership as csa_compress_fwd /
 * csa_compress_bwd; what changes is the arithmetic of the softmax weights:
 * exp is correctly rounded (the exact value rounded once to fp32), p_k =
 * e_k / den with IEEE division, and the forward sums p_k * kv_k with each
 * product and sum rounded separately, in slot order. With it, out, dkv and
 * dscore are the bits of an fp32 reference that takes those steps in that
 * order (max, exp, den, p, then the pooled sum or the backward's S); dape
 * is reduced as in csa_compress_bwd, so it is deterministic but not bitwise
 * equal to a reference that sums in another order.
 *
 * Supported only for windows of at most 8 slots (coff * ratio <= 8: ratio
 * 2, 4 or 8 with coff 1, ratio 2 or 4 with coff 2); other shapes return
 * CSA_ERR_UNSUPPORTED and launch nothing. It is slower than the default
 * mode, whose fast exp leaves a small fraction of outputs one bf16 step from
 * the eager reference.
 */
csa_status_t csa_compress_fwd_exact(const void* kv, const void* score, const float* ape,
                                    const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                                    int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                                    int32_t ratio, int32_t coff, int32_t head_dim,
                                    void* out, cudaStream_t stream);
csa_status_t csa_compress_bwd_exact(const void* kv, const void* score, const float* ape,
                                    const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                                    int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                                    int32_t ratio, int32_t coff, int32_t head_dim,
                                    const void* grad_out, void* dkv, void* dscore, float* dape,
                                    cudaStream_t stream);

/*
 * Checks the device-side preconditions on the segment arrays (the ones the
 * compute calls trust) and ORs a bit per kind of violation into *violations,
 * a caller-owned int32 in device memory that the caller zeroes first and
 * reads after synchronising the stream:
 *   CSA_SEG_BAD_START    cu_seqlens[0] != 0 or cu_seqlens_comp[0] != 0
 *   CSA_SEG_DECREASING   cu_seqlens decreases somewhere
 *   CSA_SEG_BAD_COMP     cu_seqlens_comp[s+1] - cu_seqlens_comp[s] !=
 *                        floor(seqlen_s / ratio) for some segment s
 *   CSA_SEG_PAST_END     cu_seqlens[num_seqs] > total_tokens
 *   CSA_SEG_OVER_CAPACITY cu_seqlens_comp[num_seqs] > capacity (allowed: rows
 *                        past capacity get no output slot; reported for
 *                        callers that want to know)
 * One kernel launch, asynchronous on `stream`, no host synchronisation; the
 * result is the same whatever the order the threads run in. Arguments are
 * validated as in the compute calls (num_seqs >= 1, ratio in the envelope,
 * sizes non-negative, 4-byte aligned non-null pointers).
 */
#define CSA_SEG_BAD_START 1
#define CSA_SEG_DECREASING 2
#define CSA_SEG_BAD_COMP 4
#define CSA_SEG_PAST_END 8
#define CSA_SEG_OVER_CAPACITY 16
csa_status_t csa_check_segments(const int32_t* cu_seqlens, const int32_t* cu_seqlens_comp,
                                int32_t num_seqs, int64_t total_tokens, int64_t capacity,
                                int32_t ratio, int32_t* violations, cudaStream_t stream);

/* Static description of a status code (never null). */
const char* csa_status_string(csa_status_t status);

/* The cudaError_t of the last CSA_ERR_CUDA returned on this host thread
 * (cudaSuccess if none). */
int32_t csa_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA_COMPRESS_H */
