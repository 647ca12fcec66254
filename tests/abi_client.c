/* A plain C99 client of include/csa_compress.h: it compiles against the
 * header as C (not C++), links libcsa_compress.so and drives the argument
 * validation of every entry point. Every call here is rejected or is a
 * zero-capacity no-op before any CUDA call, so it runs without a GPU.
 * Prints one line per check and exits non-zero on the first failure. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "csa_compress.h"

static int failures = 0;

static void expect(const char* what, csa_status_t got, csa_status_t want) {
  printf("%-44s %d (%s)\n", what, (int)got, csa_status_string(got));
  if (got != want) {
    printf("  expected %d\n", (int)want);
    ++failures;
  }
}

int main(void) {
  /* well-aligned addresses that are never dereferenced */
  void* a = (void*)(uintptr_t)0x10000;
  const int32_t* seg = (const int32_t*)a;
  const float* ape = (const float*)a;

  expect("fwd: ratio 3", csa_compress_fwd(a, a, ape, seg, seg, 1, 64, 8, 3, 2, 64, a, 0),
         CSA_ERR_UNSUPPORTED);
  expect("fwd: head_dim 12", csa_compress_fwd(a, a, ape, seg, seg, 1, 64, 8, 4, 2, 12, a, 0),
         CSA_ERR_UNSUPPORTED);
  expect("fwd: num_seqs 0", csa_compress_fwd(a, a, ape, seg, seg, 0, 64, 8, 4, 2, 64, a, 0),
         CSA_ERR_RANGE);
  expect("fwd: T * coff * d = 2^31",
         csa_compress_fwd(a, a, ape, seg, seg, 1, (int64_t)1 << 20, 8, 4, 2, 1024, a, 0),
         CSA_ERR_RANGE);
  expect("fwd: null kv", csa_compress_fwd(NULL, a, ape, seg, seg, 1, 64, 8, 4, 2, 64, a, 0),
         CSA_ERR_NULL);
  expect("fwd: kv 8-byte aligned",
         csa_compress_fwd((char*)a + 8, a, ape, seg, seg, 1, 64, 8, 4, 2, 64, a, 0), CSA_ERR_ALIGN);
  expect("fwd: capacity 0 launches nothing",
         csa_compress_fwd(a, a, ape, seg, seg, 1, 64, 0, 4, 2, 64, NULL, 0), CSA_OK);
  expect("bwd: null dape",
         csa_compress_bwd(a, a, ape, seg, seg, 1, 64, 8, 4, 2, 64, a, a, a, NULL, 0), CSA_ERR_NULL);
  expect("bwd_noalloc: coff 3",
         csa_compress_bwd_noalloc(a, a, ape, seg, seg, 1, 64, 8, 4, 3, 64, a, a, a, (float*)a, 0),
         CSA_ERR_UNSUPPORTED);
  expect("fwd_exact: ratio 16 (window of 16 slots)",
         csa_compress_fwd_exact(a, a, ape, seg, seg, 1, 256, 0, 16, 1, 64, NULL, 0),
         CSA_ERR_UNSUPPORTED);
  expect("fwd_exact: capacity 0 launches nothing",
         csa_compress_fwd_exact(a, a, ape, seg, seg, 1, 64, 0, 4, 2, 64, NULL, 0), CSA_OK);
  expect("bwd_exact: ratio 8, coff 2",
         csa_compress_bwd_exact(a, a, ape, seg, seg, 1, 256, 8, 8, 2, 64, a, a, a, (float*)a, 0),
         CSA_ERR_UNSUPPORTED);
  expect("check_segments: null violations word",
         csa_check_segments(seg, seg, 1, 64, 8, 4, NULL, 0), CSA_ERR_NULL);
  if (strcmp(csa_status_string((csa_status_t)99), "unknown status") != 0) ++failures;
  if (csa_last_cuda_error() != 0) ++failures;
  printf("%s\n", failures ? "FAILED" : "ok");
  return failures ? 1 : 0;
}
