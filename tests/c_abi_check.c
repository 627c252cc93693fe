/* A plain C11 caller of libds4x.so: the header compiles as C, every entry links, and the host-side
 * validation answers without a GPU (nothing here reaches a launch).  Exit status 0 = all checks
 * passed; a failed check prints its line. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "ds4x.h"

static int failures = 0;
#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      ++failures;                                                \
    }                                                            \
  } while (0)

int main(void) {
  void* A = (void*)(uintptr_t)0x10000; /* aligned, never dereferenced: validation fails first */
  const int32_t* P = (const int32_t*)A;
  CHECK(strcmp(ds4x_status_string(DS4X_OK), "DS4X_OK") == 0);
  CHECK(strncmp(ds4x_status_string(DS4X_ERR_WORKSPACE), "DS4X_ERR_WORKSPACE", 18) == 0);
  CHECK(strstr(ds4x_status_string(-42), "UNKNOWN") != NULL);

  /* sizes */
  CHECK(ds4x_workspace_bytes(2048, 2048, 512) >= (size_t)2048 * 2048 * 4);
  CHECK(ds4x_workspace_bytes(0, 2048, 512) == 0);
  CHECK(ds4x_workspace_bytes_local(2048, 2048, 512, 128) == ds4x_workspace_bytes(2048, 2048, 512));
  CHECK(ds4x_workspace_bytes_local(1, 2048, 512, DS4X_MAX_WINDOW + 1) == 0);
  CHECK(ds4x_topk_workspace_bytes(1, 262208, 512) > 0);
  CHECK(ds4x_decode_workspace_bytes(0, 512) == 0);
  CHECK(ds4x_index_and_attend_host_bytes(2048, 64, 128, 2048, 512, 64, 512, 0) > 0);
  CHECK(ds4x_index_and_attend_local_host_bytes(2048, 64, 128, 2048, 512, 64, 512, 2175, 128, 0) >
        ds4x_index_and_attend_host_bytes(2048, 64, 128, 2048, 512, 64, 512, 0));

  /* argument errors, reported before anything is launched */
  CHECK(ds4x_indexer_score(A, A, A, P, 4, 48, 128, 10, 4, (float*)A, 10, NULL) == DS4X_ERR_UNSUPPORTED);
  CHECK(ds4x_indexer_score(A, A, A, P, 4, 64, 128, 10, 4, (float*)A, 9, NULL) == DS4X_ERR_INVALID);
  CHECK(ds4x_topk((const float*)A, 10, P, 4, 10, 4, 0, (int32_t*)A, NULL, NULL, 0, NULL) == DS4X_ERR_INVALID);
  CHECK(ds4x_sparse_attn(A, A, DS4X_BF16, P, 4, 32, 512, 10, 512, 0.1f, A, NULL, NULL) == DS4X_ERR_UNSUPPORTED);
  CHECK(ds4x_index_and_attend(A, A, A, P, A, A, DS4X_BF16, 4, 64, 128, 10, 4, 512, 64, 512, 0.1f, (int32_t*)A, A,
                              NULL, NULL, 0, NULL) == DS4X_ERR_WORKSPACE);
  CHECK(ds4x_local_pooled_attn(A, A, NULL, DS4X_BF16, P, P, 4, 64, 512, 10, 512, 0, 100, 128, 0.1f, A, NULL, NULL) ==
        DS4X_ERR_INVALID);
  CHECK(ds4x_compress(A, A, (const float*)A, DS4X_F16, 16, 100, 4, NULL, NULL, 0, A, A, A, NULL) ==
        DS4X_ERR_INVALID);
  CHECK(ds4x_selftest_bounded_wait(10, NULL) == DS4X_ERR_INVALID);

  /* empty calls succeed without launching */
  CHECK(ds4x_sparse_attn(A, A, DS4X_BF16, P, 0, 64, 512, 10, 512, 0.1f, A, NULL, NULL) == DS4X_OK);
  CHECK(ds4x_compress(A, A, (const float*)A, DS4X_F16, 0, 128, 4, NULL, NULL, 0, NULL, NULL, NULL, NULL) == DS4X_OK);
  int32_t s_final = -1;
  CHECK(ds4x_decode(A, A, A, A, A, DS4X_BF16, 100, 90, A, A, 4, 359, 0, 64, 128, 4, 512, 64, 512, 0.1f,
                    (int32_t*)A, (int32_t*)A, A, NULL, A, 0, &s_final, NULL) == DS4X_OK);
  CHECK(s_final == 90);

  if (failures == 0) printf("c abi ok\n");
  return failures == 0 ? 0 : 1;
}
