// Bounded fragment planning ("[ENHANCEMENT] Shared-prefix training with
// context parallelism for exact agent trajectories", issue #7386, "Describe
// the solution you'd like": the trainer keeps fragments within a memory bound,
// repeating ancestors in several fragments where it has to; every sampled
// action keeps one loss owner).  The pages give no algorithm.  This one visits the
// segments in preorder and adds each, with whichever of its ancestors the
// current fragment lacks, while the fragment stays within the cap; otherwise
// the fragment is closed and the next starts from the segment's root path.
// A fragment owns the segments it takes in their own visit; re-added
// ancestors are context only, so each segment has exactly one owner.
#include <algorithm>
#include <vector>

#include "internal.h"

struct sp_fragments {
  int64_t physical_tokens = 0, fragment_tokens = 0;
  std::vector<int32_t> offsets, tokens, seg, owned, local_parent, local_start;
};

namespace spc {

int build_fragments(const sp_tree_desc &t, int64_t cap, sp_fragments &f) {
  const int n = t.num_segments;
  std::vector<char> in_cur(size_t(n), 0);
  std::vector<int32_t> cur_seg, cur_owned, path;
  int64_t cur_tokens = 0;
  std::vector<int32_t> local(size_t(n), -1);
  f.offsets.assign(1, 0);
  auto emit = [&]() {
    // preorder within the fragment = ascending segment id
    std::vector<int32_t> order(cur_seg.size());
    for (size_t i = 0; i < order.size(); ++i) order[i] = int32_t(i);
    std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return cur_seg[a] < cur_seg[b]; });
    const int32_t base = int32_t(f.seg.size());
    int32_t start = 0;
    for (size_t i = 0; i < order.size(); ++i) {
      const int32_t s = cur_seg[order[i]];
      local[s] = int32_t(i);
      f.seg.push_back(s);
      f.owned.push_back(cur_owned[order[i]]);
      f.local_parent.push_back(t.parent[s] >= 0 ? local[t.parent[s]] : -1);
      f.local_start.push_back(start);
      start += t.seg_len[s];
    }
    for (int32_t s : cur_seg) {
      local[s] = -1;
      in_cur[s] = 0;
    }
    f.tokens.push_back(start);
    f.fragment_tokens += start;
    f.offsets.push_back(base + int32_t(order.size()));
    cur_seg.clear();
    cur_owned.clear();
    cur_tokens = 0;
  };
  for (int s = 0; s < n; ++s) {
    path.clear();
    int64_t path_tokens = 0, extra = 0;
    for (int32_t a = s; a >= 0; a = t.parent[a]) {
      path.push_back(a);
      path_tokens += t.seg_len[a];
      if (!in_cur[a]) extra += t.seg_len[a];
    }
    if (path_tokens > cap) return SP_ERR_CAP;
    if (!cur_seg.empty() && cur_tokens + extra > cap) {
      emit();
      extra = path_tokens;
    }
    for (auto it = path.rbegin(); it != path.rend(); ++it) {
      if (in_cur[*it]) continue;
      in_cur[*it] = 1;
      cur_seg.push_back(*it);
      cur_owned.push_back(*it == s ? 1 : 0);
    }
    cur_tokens += extra;
  }
  if (!cur_seg.empty()) emit();
  f.physical_tokens = t.total_tokens;
  return SP_OK;
}

}  // namespace spc

extern "C" {

int sp_fragment_plan(const sp_tree_desc *tree, int64_t max_tokens, sp_fragments **out) {
  if (!out) return SP_ERR_INVALID_ARG;
  *out = nullptr;
  if (!tree || max_tokens < 1) return SP_ERR_INVALID_ARG;
  if (tree->num_segments < 0 || tree->total_tokens < 0) return SP_ERR_INVALID_ARG;
  if (tree->num_segments > 0 && (!tree->seg_start || !tree->seg_len || !tree->parent || !tree->depth))
    return SP_ERR_INVALID_ARG;
  if ((tree->num_segments == 0) != (tree->total_tokens == 0)) return SP_ERR_INVALID_TREE;
  if (int rc = spc::validate_tree(*tree)) return rc;
  // Each visit adds at most the segment's root path, so the entries number at
  // most the sum of (depth + 1); the tables are indexed in int32.
  int64_t bound = 0;
  for (int32_t s = 0; s < tree->num_segments; ++s) bound += int64_t(tree->depth[s]) + 1;
  if (bound > (int64_t(1) << 30)) return SP_ERR_UNSUPPORTED;
  sp_fragments *f = new (std::nothrow) sp_fragments();
  if (!f) return SP_ERR_INVALID_ARG;
  int rc = SP_OK;
  try {
    rc = spc::build_fragments(*tree, max_tokens, *f);
  } catch (...) {
    rc = SP_ERR_INVALID_ARG;
  }
  if (rc) {
    delete f;
    return rc;
  }
  *out = f;
  return SP_OK;
}

int sp_fragment_view(const sp_fragments *f, sp_fragment_info *info) {
  if (!f || !info) return SP_ERR_INVALID_ARG;
  info->num_fragments = int32_t(f->tokens.size());
  info->num_entries = int32_t(f->seg.size());
  info->physical_tokens = f->physical_tokens;
  info->fragment_tokens = f->fragment_tokens;
  info->offsets = f->offsets.data();
  info->tokens = f->tokens.data();
  info->seg = f->seg.data();
  info->owned = f->owned.data();
  info->local_parent = f->local_parent.data();
  info->local_start = f->local_start.data();
  return SP_OK;
}

void sp_fragment_destroy(sp_fragments *f) { delete f; }

}  // extern "C"
