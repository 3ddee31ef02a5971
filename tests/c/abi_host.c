/* Plain-C user of the cpkv C ABI: compiles against include/cpkv.h alone and
 * calls the host-only entry points (no GPU needed).  Prints one line per
 * check; exits non-zero on the first mismatch. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "cpkv.h"

static int fails = 0;
#define CHECK(cond, what)                              \
  do {                                                 \
    if (!(cond)) {                                     \
      printf("FAIL %s\n", what);                       \
      ++fails;                                         \
    } else {                                           \
      printf("ok %s\n", what);                         \
    }                                                  \
  } while (0)

int main(void) {
  /* two requests, page size 4: prefix 8 + 5 current tokens, prefix 0 + 4 */
  const int32_t pfx[2] = {8, 0}, cur[2] = {5, 4};
  cpkv_sizes sz;
  CHECK(cpkv_plan_sizes(2, 4, pfx, cur, &sz) == CPKV_OK, "plan_sizes returns OK");
  CHECK(sz.T == 9 && sz.C == 3 && sz.D == 5, "T=9 C=3 D=5");

  const int32_t bad_pfx[2] = {6, 0};
  CHECK(cpkv_plan_sizes(2, 4, bad_pfx, cur, &sz) == CPKV_ERR_UNALIGNED_PREFIX, "unaligned prefix rejected");
  CHECK(cpkv_plan_sizes(-1, 4, pfx, cur, &sz) == CPKV_ERR_ARG, "negative batch rejected");

  const int32_t writer[3] = {1, 0, 1};
  int64_t tpw[2];
  CHECK(cpkv_writer_token_counts(2, 4, 2, cur, writer, 3, tpw) == CPKV_OK, "writer_token_counts returns OK");
  CHECK(tpw[0] == 1 && tpw[1] == 8, "writer 0 holds 1 token, writer 1 holds 8");
  const int32_t bad_writer[3] = {1, 0, 2};
  CHECK(cpkv_writer_token_counts(2, 4, 2, cur, bad_writer, 3, tpw) == CPKV_ERR_ARG, "writer out of range rejected");

  /* ragged: q lens 6 and 4, chunk 4 -> chunk ids 0,1 (request 0), 2 (request 1) */
  const int32_t q[2] = {6, 4};
  const int32_t ci[2] = {0, 2};
  int64_t S = -1, Q = -1;
  CHECK(cpkv_ragged_plan_sizes(2, 4, q, ci, 2, &S, &Q) == CPKV_OK, "ragged_plan_sizes returns OK");
  CHECK(S == 2 && Q == 8, "two segments, 8 q tokens");
  const int32_t ci_all[3] = {0, 1, 2};
  CHECK(cpkv_ragged_plan_sizes(2, 4, q, ci_all, 3, &S, &Q) == CPKV_OK && S == 2 && Q == 10,
        "consecutive chunks of a request merge");
  const int32_t ci_bad[2] = {2, 1};
  CHECK(cpkv_ragged_plan_sizes(2, 4, q, ci_bad, 2, &S, &Q) == CPKV_ERR_ARG, "descending cp_index rejected");

  /* device entry points reject bad arguments on the host, before any launch */
  CHECK(cpkv_plan_build(2, 4, 65, 16, pfx, cur, NULL, NULL, NULL, 8, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                        NULL, NULL, NULL, 0, NULL, 0) == CPKV_ERR_ARG,
        "plan_build: cp_size above the limit rejected");
  CHECK(cpkv_plan_build(2, 4, 2, 16, pfx, cur, NULL, NULL, NULL, 4, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                        NULL, NULL, NULL, 0, NULL, 0) == CPKV_ERR_CAPACITY,
        "plan_build: dense capacity below D rejected");
  CHECK(cpkv_fill_current(2, 4, 2, 100, cur, NULL, NULL, NULL, 4, NULL, NULL, NULL, 3, 0, NULL, 0) == CPKV_ERR_ARG,
        "fill_current: row width not a multiple of 16 rejected");
  CHECK(cpkv_compose_gather_kinds(4, 1, 16, NULL, NULL, NULL, NULL, 1, 32, NULL, NULL, 0) == CPKV_ERR_ARG,
        "gather_kinds: bad kind mask rejected");
  CHECK(cpkv_compose_layer(2, 4, 2, 16, cur, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 4, NULL, 0, NULL, 0) ==
            CPKV_ERR_ARG,
        "layer compose without pointer tables rejected");

  {
    int32_t *fake = (int32_t *)(uintptr_t)256;
    int64_t *fake64 = (int64_t *)(uintptr_t)256;
    CHECK(cpkv_ragged_plan_build(2, 4, 1, 0, pfx, q, fake, 2, fake, 8, fake, fake, fake, fake, fake, fake, fake, 2,
                                 fake64, fake, 0) == CPKV_ERR_ARG,
          "ragged_plan_build: topk of 0 rejected");
  }

  CHECK(strncmp(cpkv_error_string(CPKV_ERR_CAPACITY), "CPKV_ERR_CAPACITY", 17) == 0, "error strings");
  CHECK(cpkv_version() == CPKV_VERSION, "library version matches the header");
  return fails ? 1 : 0;
}
