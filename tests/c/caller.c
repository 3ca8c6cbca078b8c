/*
 * caller.c -- a plain C99 caller of libreduce, built against
 * include/libreduce.h with no CUDA header.  It makes only calls that are
 * decided before any CUDA work (argument checks, size queries, options), so it
 * runs on a machine without a GPU, and prints one "name status" line per call
 * for the test that builds and runs it.
 */
#include <stdint.h>
#include <stdio.h>

#include "libreduce.h"

#define SHOW(name, expr) printf("%s %d\n", name, (int)(expr))

int main(void) {
  float* const fake = (float*)(uintptr_t)(1u << 20); /* never dereferenced */
  size_t bytes = 123;

  SHOW("sum_negative_n", reduce_sum_f32(fake, -1, fake, NULL));
  SHOW("sum_null_x", reduce_sum_f32(NULL, 5, fake, NULL));
  SHOW("sum_overflow", reduce_sum_f32(fake, INT64_MAX / 2, fake, NULL));
  SHOW("axis_negative", reduce_axis_f32(fake, 1, -2, 3, fake, NULL));
  SHOW("op_unknown", reduce_f32(fake, 8, fake, 9, NULL));
  SHOW("scan_bad_flags", cumsum_f32(fake, 1, 8, 1, fake + 64, 4u, NULL));
  SHOW("scan_alias", cumsum_f32(fake, 1, 8, 1, fake + 4, LIBREDUCE_SCAN_REVERSE, NULL));
  SHOW("scan_empty", cumsum_f32(fake, 0, 8, 1, fake + 64, 0u, NULL));
  SHOW("ws_query_empty", cumsum_ws_f32(fake, 3, 0, 2, fake + 64, 0u, NULL, &bytes, NULL));
  SHOW("ws_query_bytes", (int)bytes);
  SHOW("ws_null_size", reduce_axis_op_ws_f32(fake, 1, 8, 1, fake + 64, LIBREDUCE_OP_SUM, NULL, NULL, NULL));
  SHOW("option_unknown", libreduce_set_option(999, 0));
  SHOW("option_default", libreduce_set_option(LIBREDUCE_OPT_SCAN_STRATEGY, 0));
  printf("strerror_alias %s\n", libreduce_strerror(LIBREDUCE_ERR_ALIAS));
  printf("launches %lld\n", (long long)libreduce_launch_count());
  return 0;
}
