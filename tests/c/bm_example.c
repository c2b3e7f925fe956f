/* The C ABI used from C: the vLLM post's worked example ("1. overall architecture")
 * and copy-on-write example ("2.1 parallel sampling") through the host block manager.
 * Host-only calls: runs without a GPU. Prints one line per check; exits non-zero on a
 * mismatch. */
#include <stdint.h>
#include <stdio.h>

#include "pa.h"

static int fails = 0;

static void expect(int cond, const char* what) {
  printf("%s %s\n", cond ? "ok  " : "FAIL", what);
  if (!cond) ++fails;
}

int main(void) {
  /* blocks 7, 1, 3 are handed out first, as in the post's figures */
  int32_t order[16] = {7, 1, 3, 0, 2, 4, 5, 6, 8, 9, 10, 11, 12, 13, 14, 15};
  pa_bm_t bm = NULL;
  expect(pa_bm_create(16, 4, order, &bm) == PA_OK && bm != NULL, "create");
  int64_t a1 = 1, a2 = 2;
  expect(pa_bm_add(bm, a1) == PA_OK, "add A1");
  int32_t seven = 7, one = 1, n_cow = -1, src[2], dst[2];
  int64_t slots[7];
  expect(pa_bm_append(bm, &a1, &seven, 1, slots, src, dst, &n_cow) == PA_OK && n_cow == 0,
         "prompt of 7 tokens");
  const int64_t want[7] = {28, 29, 30, 31, 4, 5, 6};
  int same = 1;
  for (int i = 0; i < 7; ++i) same &= slots[i] == want[i];
  expect(same, "prompt slots 28..31, 4..6 (blocks 7 and 1)");
  expect(pa_bm_fork(bm, a1, a2) == PA_OK, "fork A1 -> A2");
  int32_t rc = 0;
  pa_bm_refcount(bm, 1, &rc);
  expect(rc == 2, "block 1 shared by both samples");
  expect(pa_bm_append(bm, &a1, &one, 1, slots, src, dst, &n_cow) == PA_OK && n_cow == 1 &&
             src[0] == 1 && dst[0] == 3 && slots[0] == 15,
         "A1 writes: copy block 1 -> 3, slot 15");
  expect(pa_bm_append(bm, &a2, &one, 1, slots, src, dst, &n_cow) == PA_OK && n_cow == 0 &&
             slots[0] == 7,
         "A2 writes in place, slot 7");
  int64_t both[2] = {1, 2};
  int32_t table[2 * 3], lens[2];
  expect(pa_bm_tables(bm, both, 2, 3, table, lens) == PA_OK && table[0] == 7 &&
             table[1] == 3 && table[2] == -1 && table[3] == 7 && table[4] == 1 &&
             lens[0] == 8 && lens[1] == 8,
         "tables A1 [7 3 -1], A2 [7 1 -1], lengths 8");
  int32_t huge = 1000;
  int32_t before = 0, after = 0;
  pa_bm_num_free(bm, &before);
  expect(pa_bm_append(bm, &a1, &huge, 1, NULL, src, dst, &n_cow) != PA_OK, "null slots refused");
  expect(pa_bm_append(bm, &a1, &huge, 1, slots, src, dst, &n_cow) == PA_ERR_NO_SPACE,
         "an append beyond the pool: PA_ERR_NO_SPACE");
  pa_bm_num_free(bm, &after);
  expect(before == after, "and nothing changed");
  expect(pa_status_string(PA_ERR_NO_SPACE)[0] != '\0', "status string");
  pa_bm_destroy(bm);
  return fails ? 1 : 0;
}
