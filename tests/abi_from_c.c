/* Drives the host-only entry points of libmoe_gb300 from plain C (C99), against the
 * public header alone: sizes, status strings and the tuning lookup.  No GPU is touched.
 * Prints one line per check; exits non-zero on the first failure. */
#include <stdio.h>
#include <string.h>

#include "moe_gb300.h"

#define CHECK(cond, msg)                    \
  do {                                      \
    if (!(cond)) {                          \
      printf("FAIL %s\n", msg);             \
      return 1;                             \
    }                                       \
    printf("ok %s\n", msg);                 \
  } while (0)

int main(void) {
  CHECK(moe_abi_version() == MOE_ABI_VERSION, "abi version matches the header");
  CHECK(strcmp(moe_status_string(MOE_OK), "ok") == 0, "status string of MOE_OK");
  /* cap = R + E (align - 1), rounded up to align */
  CHECK(moe_capacity(8192, 8, 128, 128) == 81792, "capacity of the Qwen3 layer");
  CHECK(moe_capacity(-1, 8, 128, 128) == 0, "capacity rejects T < 0");
  CHECK(moe_workspace_bytes(8192, 8, 128, 2048, 768, 128) > 0, "workspace size");
  moe_tuning_t t;
  int src = -1;
  CHECK(moe_tuning_get(4096, 3, 7, 512, 384, &t, &src) == MOE_OK && src == 0,
        "an unlisted shape takes the defaults");
  CHECK(t.swap_tails == 1 && t.da_tile_n == 256 && t.dw_chunk_rows == 4096,
        "default launch choices");
  CHECK(moe_tuning_get(8192, 8, 128, 2048, 768, NULL, &src) == MOE_ERR_INVALID_ARG,
        "NULL output is rejected");
  t.dw_chunk_rows = 100;
  CHECK(moe_tuning_override(&t) == MOE_ERR_INVALID_ARG, "out-of-range override rejected");
  t.dw_chunk_rows = 2048;
  CHECK(moe_tuning_override(&t) == MOE_OK, "override accepted");
  CHECK(moe_tuning_get(64, 2, 4, 256, 128, &t, &src) == MOE_OK && src == 2 &&
            t.dw_chunk_rows == 2048,
        "override applies to every shape");
  CHECK(moe_tuning_override(NULL) == MOE_OK, "override cleared");
  CHECK(moe_num_kernels() > 0 && moe_kernel_name(0) != NULL &&
            moe_kernel_name(moe_num_kernels()) == NULL,
        "kernel names");
  return 0;
}
