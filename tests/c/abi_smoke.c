/* A plain C99 caller of libi8lt: include/i8lt.h must compile as C, every
 * entry point used here must link, and the host-only calls must work with
 * or without a GPU.  Prints one line per check; exit status 0 when all hold.
 * Device calls are made with a null workspace so that they return an error
 * before touching any memory. */
#include <stdio.h>
#include <stdint.h>
#include <string.h>

#include "i8lt.h"

static int failures = 0;
#define CHECK(cond)                                   \
  do {                                                \
    if (!(cond)) {                                    \
      printf("FAIL %s:%d %s\n", __FILE__, __LINE__, #cond); \
      ++failures;                                     \
    }                                                 \
  } while (0)

int main(void) {
  CHECK(i8lt_abi_version() >= 2);
  CHECK(strlen(i8lt_status_string(I8LT_OK)) > 0);
  CHECK(i8lt_weight_ld(1) == 16 && i8lt_weight_ld(17) == 32);
  CHECK(i8lt_forward_workspace_size(64, 64, 64, 16) > 0);
  i8lt_fwd_layout lay;
  CHECK(i8lt_forward_workspace_layout(64, 64, 64, 16, &lay) == I8LT_OK);
  CHECK(lay.total == i8lt_forward_workspace_size(64, 64, 64, 16));
  CHECK(i8lt_backward_workspace_size(64, 64, I8LT_F16) > 0);
  CHECK(i8lt_nf4_row_bytes(100) == 64 && i8lt_nf4_blocks(100) == 2);
  float lv[16];
  CHECK(i8lt_nf4_levels(lv) == I8LT_OK);
  CHECK(lv[0] == -1.0f && lv[7] == 0.0f && lv[15] == 1.0f);
  /* argument errors come back before any device work */
  CHECK(i8lt_forward(NULL, 7, 4, 4, NULL, NULL, 4, NULL, 0, 6.0f, NULL, NULL, NULL, 0, 0, NULL, NULL) ==
        I8LT_ERR_UNSUPPORTED_DTYPE);
  CHECK(i8lt_backward_input(NULL, I8LT_F16, 4, 4, NULL, NULL, 4, NULL, NULL, NULL, 0, NULL, 0, NULL) ==
        I8LT_ERR_WORKSPACE);
  CHECK(i8lt_nf4_forward(NULL, I8LT_F32, 4, 8, NULL, NULL, 8, NULL, 0, NULL, NULL, 0, NULL) ==
        I8LT_ERR_UNSUPPORTED_DTYPE);
  printf("%s: %d failure(s)\n", failures ? "FAILED" : "ok", failures);
  return failures ? 1 : 0;
}
