/* A plain C consumer of include/gemm.h: compiled as C99 (not C++) against the header and
 * linked against the library, it runs the host-only entry points a C program uses before
 * it has a GPU: version, status strings, argument checks and the planner. Prints one line
 * per check; exits non-zero on the first failure. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "gemm.h"

#define CHECK(cond)                                                  \
  do {                                                               \
    if (!(cond)) {                                                   \
      fprintf(stderr, "FAILED: %s (line %d)\n", #cond, __LINE__);   \
      return 1;                                                      \
    }                                                                \
  } while (0)

int main(void) {
  const char *v = gemm_version();
  CHECK(v != NULL && strlen(v) > 0);
  printf("version %s\n", v);

  for (int s = GEMM_OK; s <= GEMM_ERR_DEVICE; ++s) {
    const char *msg = gemm_strerror((gemm_status_t)s);
    CHECK(msg != NULL && strlen(msg) > 0);
  }
  CHECK(gemm_strerror((gemm_status_t)12345) != NULL);

  /* the planner, without a device: bf16 8192^3, A row-major, B column-major, on 152 SMs */
  const void *a = (const void *)(uintptr_t)0x10000000u; /* aligned, never dereferenced */
  const void *b = (const void *)(uintptr_t)0x20000000u;
  void *c = (void *)(uintptr_t)0x30000000u;
  gemm_plan_info_t info;
  memset(&info, 0, sizeof info);
  gemm_status_t st = gemm_plan(NULL, 8192, 8192, 8192, a, 8192, b, 8192, c, 8192, GEMM_BF16,
                               GEMM_BF16, GEMM_PREC_DEFAULT, GEMM_ROW_MAJOR, GEMM_COL_MAJOR,
                               152, &info);
  CHECK(st == GEMM_OK);
  CHECK(info.path == GEMM_PATH_TCGEN05 && info.cta_pair == 1);
  CHECK(info.tile_m == 256 && info.tile_n == 256 && info.grid_m == 32 && info.grid_n == 32);
  printf("plan bf16 8192^3: path %d tile %dx%dx%d grid %lldx%lld ctas %lld split %d\n",
         info.path, info.tile_m, info.tile_n, info.tile_k, (long long)info.grid_m,
         (long long)info.grid_n, (long long)info.ctas, info.split_tiles);

  /* exact fp32 by default for fp32 inputs; tf32 on request */
  st = gemm_plan(NULL, 4096, 4096, 4096, a, 4096, b, 4096, c, 4096, GEMM_F32, GEMM_F32,
                 GEMM_PREC_DEFAULT, GEMM_ROW_MAJOR, GEMM_ROW_MAJOR, 152, &info);
  CHECK(st == GEMM_OK && info.path == GEMM_PATH_TCGEN05_3XTF32);
  st = gemm_plan(NULL, 4096, 4096, 4096, a, 4096, b, 4096, c, 4096, GEMM_F32, GEMM_F32,
                 GEMM_PREC_TF32, GEMM_ROW_MAJOR, GEMM_ROW_MAJOR, 152, &info);
  CHECK(st == GEMM_OK && info.path == GEMM_PATH_TCGEN05);

  /* argument errors come back synchronously */
  st = gemm_plan(NULL, 64, 64, 64, a, 32, b, 64, c, 64, GEMM_BF16, GEMM_BF16,
                 GEMM_PREC_DEFAULT, GEMM_ROW_MAJOR, GEMM_ROW_MAJOR, 152, &info);
  CHECK(st == GEMM_ERR_INVALID_ARG); /* lda < K */
  st = gemm_plan(NULL, 64, 64, 64, a, 64, b, 64, c, 64, GEMM_BF16, GEMM_BF16,
                 GEMM_PREC_TF32, GEMM_ROW_MAJOR, GEMM_ROW_MAJOR, 152, &info);
  CHECK(st == GEMM_ERR_UNSUPPORTED); /* tf32 with 16-bit inputs */
  CHECK(gemm_set_option(NULL, GEMM_OPT_GROUP_M, 8) == GEMM_ERR_INVALID_ARG);

  /* a handle needs a GPU: without one gemm_create reports the device error; with one the
   * handle is created and destroyed */
  gemm_handle_t h = NULL;
  st = gemm_create(&h, 0);
  if (st == GEMM_OK) {
    CHECK(h != NULL);
    gemm_destroy(h);
    printf("create: ok (a GPU is present)\n");
  } else {
    CHECK(st == GEMM_ERR_DEVICE || st == GEMM_ERR_CUDA);
    printf("create without a GPU: %s\n", gemm_strerror(st));
  }
  printf("all checks passed\n");
  return 0;
}
