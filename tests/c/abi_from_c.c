/* Drives the library's host-side entry points from plain C99: planning, the plan
 * view, fragment planning, argument errors and status strings.  No GPU call.
 *
 * stdin:  n, then n lines "seg_start seg_len parent depth", then
 *         "tile_tokens kv_block order fragment_cap".
 * stdout: the plan and fragment tables as text lines (read by the Python test,
 *         which compares them with the oracle). */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "shared_prefix_causal.h"

static int fail(const char *what) {
  fprintf(stderr, "abi_from_c: %s\n", what);
  return 1;
}

int main(void) {
  int n = 0;
  if (scanf("%d", &n) != 1 || n < 0) return fail("bad tree header");
  int32_t *buf = (int32_t *)calloc((size_t)(4 * n + 1), sizeof(int32_t));
  if (!buf) return fail("out of memory");
  int32_t *start = buf, *len = buf + n, *parent = buf + 2 * n, *depth = buf + 3 * n;
  int64_t total = 0;
  for (int s = 0; s < n; ++s) {
    if (scanf("%d %d %d %d", &start[s], &len[s], &parent[s], &depth[s]) != 4) return fail("bad segment line");
    total += len[s];
  }
  int tile = 0, kvb = 0, order = 0;
  long long cap = 0;
  if (scanf("%d %d %d %lld", &tile, &kvb, &order, &cap) != 4) return fail("bad plan line");

  sp_tree_desc tree;
  tree.num_segments = n;
  tree.total_tokens = (int32_t)total;
  tree.seg_start = start;
  tree.seg_len = len;
  tree.parent = parent;
  tree.depth = depth;

  /* argument errors come back as statuses, and *out is cleared */
  sp_plan *p = (sp_plan *)&tree; /* any non-null value: must be overwritten with NULL */
  if (sp_tree_plan(NULL, tile, kvb, order, &p) != SP_ERR_INVALID_ARG || p != NULL) return fail("null tree");
  if (sp_tree_plan(&tree, tile, kvb, order, NULL) != SP_ERR_INVALID_ARG) return fail("null out");
  if (sp_tree_plan(&tree, 0, kvb, order, &p) != SP_ERR_INVALID_ARG || p != NULL) return fail("tile 0");
  if (sp_plan_view(NULL, NULL) != SP_ERR_INVALID_ARG) return fail("null view");
  sp_plan_destroy(NULL);
  sp_fragment_destroy(NULL);
  tree.total_tokens = (int32_t)(total + 1); /* lengths no longer add up to the token count */
  if (sp_tree_plan(&tree, tile, kvb, order, &p) != SP_ERR_INVALID_TREE || p != NULL) return fail("wrong total");
  tree.total_tokens = (int32_t)total;
  for (int code = 0; code >= -10; --code) {
    const char *msg = sp_status_string(code);
    if (!msg || !msg[0]) return fail("empty status string");
  }

  int rc = sp_tree_plan(&tree, tile, kvb, order, &p);
  sp_plan_info info;
  memset(&info, 0, sizeof info);
  if (rc == SP_OK && sp_plan_view(p, &info) != SP_OK) return fail("view");
  printf("plan %d %d %d %d %d\n", rc, info.n_tiles, info.n_ranges, info.n_bwd, info.max_ranges_per_tile);
  for (int i = 0; i < info.n_tiles; ++i) {
    const int32_t *t = info.tiles + 5 * i;
    printf("T %d %d %d %d %d\n", t[0], t[1], t[2], t[3], t[4]);
  }
  for (int i = 0; i < info.n_ranges; ++i) printf("R %d %d\n", info.ranges[2 * i], info.ranges[2 * i + 1]);
  for (int i = 0; i < info.n_bwd; ++i) {
    const int32_t *b = info.bwd + 5 * i;
    printf("B %d %d %d %d %d\n", b[0], b[1], b[2], b[3], b[4]);
  }
  if (rc == SP_OK) {
    const int32_t *rows = NULL, *key_end = NULL;
    int32_t n_rows = 0;
    if (sp_plan_bwd_blocks(NULL, &rows, &n_rows, &key_end) != SP_ERR_INVALID_ARG) return fail("null bwd blocks");
    if (sp_plan_bwd_blocks(p, &rows, &n_rows, &key_end) != SP_OK) return fail("bwd blocks");
    for (int i = 0; i < n_rows; ++i) {
      const int32_t *b = rows + 5 * i;
      printf("M %d %d %d %d %d\n", b[0], b[1], b[2], b[3], b[4]);
    }
    printf("E");
    for (int i = 0; i < info.total_tokens; ++i) printf(" %d", key_end[i]);
    printf("\n");
  }
  sp_plan_destroy(p);

  sp_fragments *fr = NULL;
  rc = sp_fragment_plan(&tree, (int64_t)cap, &fr);
  sp_fragment_info fi;
  memset(&fi, 0, sizeof fi);
  if (rc == SP_OK && sp_fragment_view(fr, &fi) != SP_OK) return fail("fragment view");
  printf("frag %d %d %d %lld %lld\n", rc, fi.num_fragments, fi.num_entries, (long long)fi.physical_tokens,
         (long long)fi.fragment_tokens);
  for (int f = 0; f <= fi.num_fragments && rc == SP_OK; ++f) printf("O %d\n", fi.offsets[f]);
  for (int e = 0; e < fi.num_entries; ++e)
    printf("F %d %d %d %d\n", fi.seg[e], fi.owned[e], fi.local_parent[e], fi.local_start[e]);
  sp_fragment_destroy(fr);
  free(buf);
  return 0;
}
