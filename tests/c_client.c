/* A plain C99 client of include/w4a16.h: it compiles against the header
 * alone, links the shared library, and calls the entry points that need no
 * GPU (size queries, argument checks, status strings, switches). Exit status
 * 0 when every check holds; the first failure is printed. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "w4a16.h"

static int failures = 0;

#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__,     \
              __LINE__, #cond);                                  \
      ++failures;                                                \
    }                                                            \
  } while (0)

int main(void) {
  /* an aligned, non-null address that the argument checks never follow */
  void *const fake = (void *)(uintptr_t)(1u << 20);
  uint16_t *const fx = (uint16_t *)fake;

  /* N = 256, K = 512, G = 128: 16 tiles x 8 chunks x 512 B of codes, one
   * 4-group block of scales per tile (128 B), zero points 32 B per tile */
  CHECK(w4a16_repacked_bytes(256, 512, 128, W4A16_SYMMETRIC) == 65536 + 2048);
  CHECK(w4a16_repacked_bytes(256, 512, 128, W4A16_ZERO_POINTS) == 65536 + 2048 + 512);
  /* affine: biases in the scales' layout, then the bias operand of 256 rows
   * x 64 bf16 columns (3 x 4 groups rounded up to 64) */
  CHECK(w4a16_repacked_bytes(256, 512, 128, W4A16_AFFINE) == 65536 + 2048 + 2048 + 256 * 64 * 2);
  CHECK(w4a16_gateup_repacked_bytes(100, 512, 128, W4A16_SYMMETRIC) ==
        w4a16_repacked_bytes(256, 512, 128, W4A16_SYMMETRIC));
  CHECK(w4a16_repacked_bytes(256, 512, 96, W4A16_SYMMETRIC) == 0);
  CHECK(w4a16_repacked_bytes(256, 512, 128, 3) == 0);
  CHECK(w4a16_xsum_bytes(4, 5120, 64) == 4 * 256 * 2);
  CHECK(w4a16_xsum_bytes(0, 5120, 64) == 0);

  /* argument checks return before any CUDA call */
  CHECK(w4a16_gemm(NULL, fake, NULL, NULL, 4, 64, 128, 64, W4A16_SYMMETRIC, fx, NULL) ==
        W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemm(fx, fake, fake, NULL, 4, 64, 128, 64, W4A16_SYMMETRIC, fx, NULL) ==
        W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemm(fx, fake, NULL, NULL, 4, 64, 96, 64, W4A16_SYMMETRIC, fx, NULL) ==
        W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemm(fx, fake, NULL, NULL, 4, 64, 128, 64, W4A16_AFFINE, fx, NULL) ==
        W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemm(fx + 4, fake, NULL, NULL, 4, 64, 128, 64, W4A16_SYMMETRIC, fx, NULL) ==
        W4A16_ERR_MISALIGNED);
  CHECK(w4a16_gateup_silu(fx, NULL, 4, 64, 128, 64, W4A16_SYMMETRIC, fx, NULL) ==
        W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemm_argmax(fx, fake, 33, 64, 128, 64, W4A16_SYMMETRIC, NULL, (int64_t *)fake, NULL) ==
        W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemm_affine(fx, NULL, fake, 33, 64, 128, 64, fx, NULL) == W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_gemm_affine_noalloc(fx, fake, 8193, 64, 5120, 64, fx, NULL) == W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_xsum(fx, 4, 128, 64, NULL, NULL) == W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_repack(NULL, (const uint16_t *)fake, NULL, 64, 128, 64, W4A16_SYMMETRIC, fake, NULL) ==
        W4A16_ERR_INVALID_ARG);
  CHECK(w4a16_dequantize(fake, 64, 128, 48, W4A16_SYMMETRIC, (float *)fake, NULL) == W4A16_ERR_INVALID_ARG);

  /* status strings and switches */
  CHECK(w4a16_strerror(W4A16_OK) != NULL && strlen(w4a16_strerror(W4A16_OK)) > 0);
  CHECK(strcmp(w4a16_strerror(-99), "unknown status") == 0);
  {
    int prev = w4a16_set_kernel_override(2);
    CHECK(prev >= 0 && prev <= 4);
    CHECK(w4a16_set_kernel_override(prev) == 2);
    CHECK(w4a16_set_kernel_override(7) == -1);
  }
  {
    int prev = w4a16_set_programmatic_overlap(1);
    CHECK(prev == 0 || prev == 1);
    CHECK(w4a16_set_programmatic_overlap(prev) == 1);
    CHECK(w4a16_set_programmatic_overlap(2) == -1);
  }

  if (failures) return 1;
  printf("c client ok\n");
  return 0;
}
