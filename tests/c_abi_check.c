/* A plain C (C11) caller of the library's host-side entry points: the header compiles as C and the
 * symbols link without C++ or Python.  Prints one "name value" line per check; exits non-zero on a
 * failed expectation.  Built and run by tests/test_c_abi.py (no GPU needed). */
#include <stdio.h>
#include <string.h>

#include "rdkv.h"

static int fails = 0;
static void expect(int ok, const char* what) {
  if (!ok) {
    fprintf(stderr, "FAILED: %s (%s)\n", what, rdkv_last_error_string());
    ++fails;
  }
}

int main(void) {
  rdkv_shape s = {1, 32768, 24, 8, 128, 128, RDKV_F16};
  printf("version %d\n", (int)rdkv_version());
  const size_t ws_score = rdkv_workspace_bytes(&s, RDKV_CALL_SCORE);
  const size_t ws_alloc = rdkv_workspace_bytes(&s, RDKV_CALL_ALLOCATE);
  printf("ws_score %zu\nws_alloc %zu\nplan_bytes %zu\n", ws_score, ws_alloc, rdkv_plan_bytes(&s));
  expect(ws_score == rdkv_score_workspace_bytes(&s), "score workspace query");
  expect(ws_alloc == rdkv_allocate_workspace_bytes(&s), "allocate workspace query");

  rdkv_sizes b;
  memset(&b, 0, sizeof(b));
  expect(rdkv_zone_bounds(&s, 2.5f, 2.5f, &b) == RDKV_OK, "zone bounds");
  printf("bound_zone_a %lld\nbound_index_slots %lld\nbound_n_heads %d\n", (long long)b.zone_a_bytes,
         (long long)b.index_slots, (int)b.n_heads);
  expect(b.zone_a_bytes > 0 && b.index_slots > 0 && b.n_heads == 8, "bound values");

  const size_t ws_ap = rdkv_allocate_pack_workspace_bytes(&s, 0);
  printf("ws_allocate_pack %zu\n", ws_ap);
  expect(ws_ap > 0 && rdkv_allocate_pack_workspace_bytes(&s, 1) >= ws_ap, "allocate+pack workspace query");
  expect(rdkv_allocate_pack_workspace_bytes(&s, 2) == 0, "allocate+pack scope checked");

  rdkv_shape bad = s;
  bad.head_dim = 96;
  const rdkv_status st = rdkv_zone_bounds(&bad, 2.5f, 2.5f, &b);
  printf("bad_head_dim_status %d\n", (int)st);
  expect(st == RDKV_ERR_UNSUPPORTED, "unsupported head_dim refused");
  expect(strlen(rdkv_last_error_string()) > 0, "error message set");
  return fails == 0 ? 0 : 1;
}
