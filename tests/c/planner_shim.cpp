// The host planner (plan.cpp) behind a plain C interface, for tests that build
// plan.cpp and fragments.cpp on their own with g++ (no CUDA).  The fragment
// planner's own extern "C" entry points are used as they are.
#include "internal.h"

extern "C" {

SP_API void *shim_plan(const sp_tree_desc *t, int32_t tile, int32_t kvb, int32_t order, int32_t *rc) {
  sp_plan *p = new sp_plan();
  *rc = spc::build_plan(*t, tile, kvb, order, *p);
  if (*rc != SP_OK) {
    delete p;
    return nullptr;
  }
  return p;
}

// Builds the tables the kernels read (forward tile pairs and quads with their
// merged 128-key block lists; the backward launch order), as the first upload
// does.
SP_API void shim_device_tables(void *h) {
  sp_plan *p = static_cast<sp_plan *>(h);
  spc::build_pairs(*p, 128);
  spc::build_quads(*p, 128);
  spc::build_bwd_schedule(*p);
}

SP_API int64_t shim_bwd_run_sum(void *h) { return static_cast<const sp_plan *>(h)->bwd_run_sum; }
SP_API int32_t shim_bwd_run_max(void *h) { return static_cast<const sp_plan *>(h)->bwd_run_max; }
SP_API int64_t shim_bwdm_run_sum(void *h) { return static_cast<const sp_plan *>(h)->bwdm_run_sum; }
SP_API int32_t shim_bwdm_run_max(void *h) { return static_cast<const sp_plan *>(h)->bwdm_run_max; }

// which: 0 tiles [n][5], 1 ranges [n][2], 2 bwd [n][5], 3 pairs [n][4],
// 4 pblk [n][8], 5 bwd_sched [n][5], 6 quads [n][6], 7 qblk [n][8],
// 8 bwd_merged [n][5], 9 key_end [n][1]; returns the row count
SP_API int32_t shim_rows(void *h, int32_t which, const int32_t **data) {
  const sp_plan *p = static_cast<const sp_plan *>(h);
  static const int width[10] = {5, 2, 5, 4, 8, 5, 6, 8, 5, 1};
  const std::vector<int32_t> *tables[10] = {&p->tiles, &p->ranges,    &p->bwd,   &p->pairs,      &p->pblk,
                                            &p->bwd_sched, &p->quads, &p->qblk, &p->bwd_merged, &p->key_end};
  const std::vector<int32_t> &v = *tables[which];
  *data = v.data();
  return int32_t(v.size() / width[which]);
}

SP_API void shim_free(void *h) { delete static_cast<sp_plan *>(h); }

// merge_runs on arbitrary run lists: lists holds count[i] runs {kb, nb, end,
// causal} per slot i, one after another; writes up to cap entries of 8 int32
// and returns the entry count.
SP_API int32_t shim_merge_runs(const int32_t *lists, const int32_t *count, int32_t block_keys, int32_t *out,
                               int32_t cap) {
  std::vector<spc::TileRun> l[4];
  for (int i = 0; i < 4; ++i)
    for (int32_t r = 0; r < count[i]; ++r, lists += 4) l[i].push_back({lists[0], lists[1], lists[2], lists[3] != 0});
  std::vector<int32_t> runs;
  const int32_t n = spc::merge_runs(l, block_keys, runs);
  for (int32_t i = 0; i < n && i < cap; ++i)
    for (int j = 0; j < 8; ++j) out[8 * i + j] = runs[8 * size_t(i) + j];
  return n;
}

}  // extern "C"
