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

// which: 0 tiles [n][5], 1 ranges [n][2], 2 bwd [n][5]; returns the row count
SP_API int32_t shim_rows(void *h, int32_t which, const int32_t **data) {
  const sp_plan *p = static_cast<const sp_plan *>(h);
  const std::vector<int32_t> &v = which == 0 ? p->tiles : which == 1 ? p->ranges : p->bwd;
  *data = v.data();
  return int32_t(v.size() / (which == 1 ? 2 : 5));
}

SP_API void shim_free(void *h) { delete static_cast<sp_plan *>(h); }

}  // extern "C"
