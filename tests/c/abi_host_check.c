/* A plain C99 caller of the segkv C ABI, run without a GPU: a host-only
 * handle (no pools) plans and tracks pages but launches nothing. It checks
 * that include/segkv.h compiles as C and that the calls behave as declared:
 * kept ranges after append and trim, page counts, a decode plan's key
 * coverage, and the error codes of refused calls. Exit status 0 = pass. */
#include <stdio.h>
#include <string.h>

#include "segkv.h"

#define CHECK(c)                                                  \
  do {                                                            \
    if (!(c)) {                                                   \
      fprintf(stderr, "abi_host_check line %d: %s\n", __LINE__, #c); \
      return 1;                                                   \
    }                                                             \
  } while (0)

static int run(segkv_t* hp) {
  /* one layer, 8 query / 2 KV heads of 64 dims; KV head 0 global, 1 local
   * with a window of 16 keys; pages of 16 tokens */
  const uint8_t cls[2] = {SEGKV_GLOBAL, SEGKV_LOCAL};
  const int32_t win[1] = {16};
  const int32_t ids[1] = {0};
  segkv_stats_t st, st2;
  int32_t start = -1, len = -1, first = -1, pids[16], nids = -1;
  segkv_t h;

  CHECK(segkv_create(hp, 1, 8, 2, 64, cls, win, 16, 2, 256, NULL, NULL, 64, 0.f) == SEGKV_OK);
  h = *hp;

  /* 100 tokens: every head keeps all of them (the chunk's queries need them) */
  {
    const int32_t cu[2] = {0, 100};
    CHECK(segkv_append(h, 0, NULL, NULL, cu, ids, 1, NULL) == SEGKV_OK);
  }
  CHECK(segkv_stats(h, &st) == SEGKV_OK);
  CHECK(st.num_pages == 64 && st.pages_global == 7 && st.pages_local == 7);
  CHECK(st.pages_in_use == 14 && st.kept_tokens == 200);

  /* trim: the local head keeps [100 - 16 + 1, 100) = [85, 100), whole pages
   * 5 and 6; pages 0..4 end at or below 85 and are freed */
  CHECK(segkv_trim(h, 0, ids, 1) == SEGKV_OK);
  CHECK(segkv_stats(h, &st) == SEGKV_OK);
  CHECK(st.pages_global == 7 && st.pages_local == 2 && st.kept_tokens == 115);
  CHECK(segkv_get_segment(h, 0, 1, 0, &start, &len, &first, pids, 16, &nids) == SEGKV_OK);
  CHECK(start == 85 && len == 15 && first == 5 && nids == 2);
  CHECK(segkv_get_segment(h, 0, 0, 0, &start, &len, &first, pids, 16, &nids) == SEGKV_OK);
  CHECK(start == 0 && len == 100 && first == 0 && nids == 7);

  /* the next token, then the plan of its decode over 4 CTAs: the global head
   * streams keys [0, 101), the local head [85, 101), each key once */
  {
    const int32_t cu[2] = {0, 1};
    const int32_t lens[1] = {101};
    int32_t units[8 * 64], cta[9], covered[2] = {0, 0};
    int nu = 0, nc = 0, u, prev_end[2] = {-1, -1};
    CHECK(segkv_append(h, 0, NULL, NULL, cu, ids, 1, NULL) == SEGKV_OK);
    CHECK(segkv_plan_decode(h, 0, 1, lens, ids, 1, 4, units, 64, cta, 8, &nu, &nc) == SEGKV_OK);
    CHECK(nu >= 2 && nc >= 1 && nc <= 4 && cta[0] == 0 && cta[nc] == nu);
    for (u = 0; u < nu; ++u) {
      const int32_t* x = units + 8 * u;
      const int hd = x[1];
      CHECK(x[0] == 0 && (hd == 0 || hd == 1) && x[2] == hd && x[7] == 100);
      CHECK(x[4] > x[3]);
      CHECK(prev_end[hd] < 0 ? x[3] == (hd ? 85 : 0) : x[3] == prev_end[hd]);
      prev_end[hd] = x[4];
      covered[hd] += x[4] - x[3];
    }
    CHECK(prev_end[0] == 101 && prev_end[1] == 101 && covered[0] == 101 && covered[1] == 16);

    /* three query tokens would need key 83 of the local head: evicted */
    CHECK(segkv_plan_decode(h, 0, 3, lens, ids, 1, 4, units, 64, cta, 8, &nu, &nc) ==
          SEGKV_ERR_EVICTED);
  }

  /* refused calls return their code, record a message and change nothing */
  CHECK(segkv_stats(h, &st) == SEGKV_OK);
  {
    const int32_t cu[2] = {0, 1};
    const int32_t bad_ids[1] = {7};
    size_t ws = 0;
    CHECK(segkv_append(h, 1, NULL, NULL, cu, ids, 1, NULL) == SEGKV_ERR_INVALID_ARG);
    CHECK(strlen(segkv_last_error(h)) > 0);
    CHECK(segkv_append(h, 0, NULL, NULL, cu, bad_ids, 1, NULL) == SEGKV_ERR_INVALID_ARG);
    CHECK(segkv_decode_attn(h, 0, NULL, cu, ids, 1, NULL, NULL, 0, NULL) == SEGKV_ERR_INVALID_ARG);
    CHECK(segkv_workspace_size(h, SEGKV_WS_DECODE, 1, 1, &ws) == SEGKV_OK && ws > 0);
  }
  CHECK(segkv_stats(h, &st2) == SEGKV_OK);
  CHECK(memcmp(&st, &st2, sizeof st) == 0);

  /* freeing the sequence returns every page */
  CHECK(segkv_free_seq(h, 0) == SEGKV_OK);
  CHECK(segkv_stats(h, &st) == SEGKV_OK);
  CHECK(st.pages_in_use == 0 && st.kept_tokens == 0);
  return 0;
}

int main(void) {
  segkv_t h = NULL;
  const int rc = run(&h);
  if (h) {
    if (segkv_destroy(h) != SEGKV_OK) return 1;
  }
  if (rc == 0) printf("ok\n");
  return rc;
}
