// Host planner: tree validation and the per-query-tile ancestor KV-range
// lists ("[ENHANCEMENT] Shared-prefix training with context parallelism for
// exact agent trajectories", issue #7386, "Describe the solution you'd like":
// every query run attends to its ancestor path only; PR #7387
// "TreePackedSeqParams", "Summary": a query segment attends causally over its
// ancestors).
//
// One preorder pass with an explicit root-path stack validates the tree and
// builds, per segment, the merged token intervals of its root path; a reverse
// pass gives each segment's subtree end.  Tiles and backward blocks are then
// emitted and sorted.  The canonical output (tile order, range merging,
// backward order) is documented in the public header.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <numeric>
#include <utility>
#include <vector>

#include "internal.h"

namespace spc {
namespace {

using Interval = std::pair<int32_t, int32_t>;

// Largest number of root-path intervals, or of tile ranges, a plan may hold
// (its tables are indexed in int32).
constexpr int64_t kMaxEntries = int64_t(1) << 30;

int validate_impl(const sp_tree_desc &t) {
  const int n = t.num_segments;
  int64_t pos = 0;
  for (int s = 0; s < n; ++s) {
    if (t.seg_len[s] < 1 || t.seg_start[s] != pos) return SP_ERR_INVALID_TREE;
    pos += t.seg_len[s];
  }
  if (pos != t.total_tokens) return SP_ERR_INVALID_TREE;
  std::vector<int32_t> stack;  // root path of the last placed segment
  for (int s = 0; s < n; ++s) {
    const int32_t p = t.parent[s];
    if (p < -1 || p >= s) return SP_ERR_INVALID_TREE;
    if (t.depth[s] != (p < 0 ? 0 : t.depth[p] + 1)) return SP_ERR_INVALID_TREE;
    if (p < 0) {
      stack.clear();
    } else {
      while (!stack.empty() && stack.back() != p) stack.pop_back();
      if (stack.empty()) return SP_ERR_INVALID_TREE;  // parent's subtree already closed
    }
    stack.push_back(s);
  }
  return SP_OK;
}

}  // namespace

int validate_tree(const sp_tree_desc &t) { return validate_impl(t); }

int build_plan(const sp_tree_desc &t, int32_t tile_tokens, int32_t kv_block, int32_t order,
               sp_plan &plan) {
  if (tile_tokens <= 0 || kv_block <= 0 || (order != 0 && order != 1)) return SP_ERR_INVALID_ARG;
  if (t.num_segments < 0 || t.total_tokens < 0) return SP_ERR_INVALID_ARG;
  if (t.num_segments > 0 &&
      (!t.seg_start || !t.seg_len || !t.parent || !t.depth))
    return SP_ERR_INVALID_ARG;
  if ((t.num_segments == 0) != (t.total_tokens == 0)) return SP_ERR_INVALID_TREE;
  if (int rc = validate_impl(t)) return rc;

  const int n = t.num_segments;
  plan.tile_tokens = tile_tokens;
  plan.kv_block = kv_block;
  plan.order = order;
  plan.total_tokens = t.total_tokens;
  plan.num_segments = n;

  // Intervals of each segment's root path: the parent's, then the segment
  // itself, merged into the parent's last interval when it starts where that
  // one ends (a first child, placed right after its parent).  A tile's ranges
  // are its segment's root path cut at the tile's end, so they number the
  // same.  Both totals are counted first: the plan's tables are indexed in
  // int32, and a tree whose tables would pass kMaxEntries entries (possible
  // for deep trees whose paths do not merge) is refused before anything is
  // allocated.
  std::vector<int32_t> path_len(n);
  std::vector<char> merges(n);
  int64_t pool_total = 0, range_total = 0;
  for (int s = 0; s < n; ++s) {
    const int32_t p = t.parent[s];
    merges[s] = p >= 0 && t.seg_start[p] + t.seg_len[p] == t.seg_start[s];
    path_len[s] = (p >= 0 ? path_len[p] : 0) + (merges[s] ? 0 : 1);
    pool_total += path_len[s];
    range_total += (int64_t(t.seg_len[s]) + tile_tokens - 1) / tile_tokens * path_len[s];
  }
  if (pool_total > kMaxEntries || range_total > kMaxEntries) return SP_ERR_UNSUPPORTED;
  std::vector<Interval> pool;
  pool.reserve(size_t(pool_total));
  std::vector<int32_t> path_off(size_t(n) + 1, 0), root(n), send(n);
  std::vector<int64_t> anc_tokens(n, 0);
  for (int s = 0; s < n; ++s) {
    const int32_t p = t.parent[s], a0 = t.seg_start[s], a1 = a0 + t.seg_len[s];
    path_off[s] = int32_t(pool.size());
    if (p >= 0) {
      pool.insert(pool.end(), pool.begin() + path_off[p], pool.begin() + path_off[p + 1]);
      anc_tokens[s] = anc_tokens[p] + t.seg_len[p];
    }
    if (merges[s])
      pool.back().second = a1;
    else
      pool.push_back({a0, a1});
    path_off[s + 1] = int32_t(pool.size());
    root[s] = p < 0 ? s : root[p];
    send[s] = a1;
  }
  for (int s = n - 1; s >= 0; --s)
    if (t.parent[s] >= 0) send[t.parent[s]] = std::max(send[t.parent[s]], send[s]);

  // A tile reads its parent's root path, then its own segment up to the
  // tile's end (merged into the last interval when they touch).
  struct Tile {
    int32_t seg, k, q0, q1;
    int64_t kv_total;
  };
  size_t n_tiles = 0;
  for (int s = 0; s < n; ++s) n_tiles += size_t((int64_t(t.seg_len[s]) + tile_tokens - 1) / tile_tokens);
  std::vector<Tile> tiles;
  tiles.reserve(n_tiles);
  for (int s = 0; s < n; ++s) {
    const int32_t a0 = t.seg_start[s], a1 = a0 + t.seg_len[s];
    int32_t k = 0;
    for (int32_t q0 = a0; q0 < a1; q0 += tile_tokens, ++k) {
      const int32_t q1 = std::min(a1, q0 + tile_tokens);
      tiles.push_back({s, k, q0, q1, anc_tokens[s] + (q1 - a0)});
    }
  }
  // Sort keys as two integers compared in order; every field is non-negative
  // and below 2^31, so each pair of fields packs into one int64 without
  // changing the order.  Order 0: (root, parent + 1) then (tile index,
  // segment); order 1: (-kv_total) then (segment, tile index).
  struct Key {
    int64_t a, b;
    int32_t tile;
  };
  std::vector<Key> keys(tiles.size());
  for (size_t i = 0; i < tiles.size(); ++i) {
    const Tile &x = tiles[i];
    if (order == 0)
      keys[i] = {(int64_t(root[x.seg]) << 32) | int64_t(t.parent[x.seg] + 1), (int64_t(x.k) << 32) | x.seg,
                 int32_t(i)};
    else
      keys[i] = {-x.kv_total, (int64_t(x.seg) << 32) | x.k, int32_t(i)};
  }
  std::sort(keys.begin(), keys.end(), [](const Key &x, const Key &y) { return x.a != y.a ? x.a < y.a : x.b < y.b; });
  plan.tiles.clear();
  plan.ranges.clear();
  plan.tiles.reserve(5 * tiles.size());
  plan.ranges.reserve(2 * size_t(range_total));
  plan.max_ranges_per_tile = 0;
  for (const Key &key : keys) {
    const Tile &x = tiles[key.tile];
    const int32_t p = t.parent[x.seg], a0 = t.seg_start[x.seg];
    const int32_t rb = int32_t(plan.ranges.size() / 2);
    if (p >= 0)
      for (int32_t j = path_off[p]; j < path_off[p + 1]; ++j) {
        plan.ranges.push_back(pool[j].first);
        plan.ranges.push_back(pool[j].second);
      }
    if (!plan.ranges.empty() && int32_t(plan.ranges.size() / 2) > rb && plan.ranges.back() == a0) {
      plan.ranges.back() = x.q1;
    } else {
      plan.ranges.push_back(a0);
      plan.ranges.push_back(x.q1);
    }
    const int32_t rc = int32_t(plan.ranges.size() / 2) - rb;
    for (int32_t v : {x.seg, x.q0, x.q1, rb, rc}) plan.tiles.push_back(v);
    plan.max_ranges_per_tile = std::max(plan.max_ranges_per_tile, rc);
  }

  struct Blk {
    int32_t seg, k0, k1, q0, q1;
  };
  std::vector<Blk> blocks;
  for (int s = 0; s < n; ++s) {
    const int32_t a0 = t.seg_start[s], a1 = a0 + t.seg_len[s];
    for (int32_t k0 = a0; k0 < a1; k0 += kv_block)
      blocks.push_back({s, k0, std::min(a1, k0 + kv_block), k0, send[s]});
  }
  std::sort(blocks.begin(), blocks.end(), [](const Blk &x, const Blk &y) {
    const int32_t cx = x.q1 - x.q0, cy = y.q1 - y.q0;
    if (cx != cy) return cx > cy;
    return x.k0 < y.k0;
  });
  plan.bwd.clear();
  for (auto &b : blocks) plan.bwd.insert(plan.bwd.end(), {b.seg, b.k0, b.k1, b.q0, b.q1});
  return SP_OK;
}

namespace {

void tile_runs(const sp_plan &plan, int32_t t, int32_t block_keys, std::vector<TileRun> &out) {
  out.clear();
  if (t < 0) return;
  const int32_t *tl = &plan.tiles[5 * size_t(t)];
  for (int32_t r = 0; r < tl[4]; ++r) {
    const int32_t a = plan.ranges[2 * size_t(tl[3] + r)], e = plan.ranges[2 * size_t(tl[3] + r) + 1];
    out.push_back({a, int32_t((int64_t(e) - a + block_keys - 1) / block_keys), e, r + 1 == tl[4]});
  }
}

}  // namespace

// Merges the block lists of up to four tiles (absent: an empty list) by block
// start and appends the result to `runs` as entries of 8 int32
//   {kb, nb, end[0], end[1], end[2], end[3], causal bits, 0}:
// nb blocks starting at kb, kb + B, ..., each read by exactly the tiles i with
// end[i] != 0 (up to end[i]; bit i set where that is tile i's causal range).
// Expanded block by block this is the list that merges equal block starts of
// the tiles' lists; a run stops where another tile's next block would start
// inside it, so tiles share an entry only where their blocks start at the
// same key.  Returns the number of entries.
int32_t merge_runs(std::vector<TileRun> (&lists)[4], int32_t block_keys, std::vector<int32_t> &runs) {
  constexpr int64_t kNone = INT64_MAX;
  size_t ri[4] = {0, 0, 0, 0};
  int64_t bi[4] = {0, 0, 0, 0};
  auto cur = [&](int i) -> int64_t {
    return ri[i] < lists[i].size() ? int64_t(lists[i][ri[i]].kb) + int64_t(block_keys) * bi[i] : kNone;
  };
  int32_t count = 0;
  for (;;) {
    int64_t kb = kNone;
    for (int i = 0; i < 4; ++i) kb = std::min(kb, cur(i));
    if (kb == kNone) break;
    int64_t n = kNone;
    int32_t e[4] = {0, 0, 0, 0}, flags = 0;
    for (int i = 0; i < 4; ++i) {
      const int64_t c = cur(i);
      if (c == kb) {
        const TileRun &tr = lists[i][ri[i]];
        n = std::min(n, int64_t(tr.nb) - bi[i]);
        e[i] = tr.end;
        flags |= tr.causal ? (1 << i) : 0;
      } else if (c != kNone) {
        n = std::min(n, (c - kb + block_keys - 1) / block_keys);  // stop before tile i's next block
      }
    }
    runs.insert(runs.end(), {int32_t(kb), int32_t(n), e[0], e[1], e[2], e[3], flags, 0});
    ++count;
    for (int i = 0; i < 4; ++i)
      if (e[i] != 0 && (bi[i] += n) == lists[i][ri[i]].nb) {
        ++ri[i];
        bi[i] = 0;
      }
  }
  return count;
}

// Pairs tiles (2i, 2i+1) in schedule order -- tile k of sibling segments, or
// neighbouring tiles of one segment -- and merges their key blocks by start
// (tile a in slot 0, tile b in slot 1 of each run).  Shared ancestor blocks
// then appear once, so one K/V load feeds both tiles; a run covers a whole
// stretch of blocks both tiles read alike, so the table grows with the
// number of ranges, not of key blocks.
void build_pairs(sp_plan &plan, int32_t block_keys) {
  plan.pairs.clear();
  plan.pblk.clear();
  const int32_t nt = plan.n_tiles();
  std::vector<TileRun> lists[4];
  for (int32_t t = 0; t < nt; t += 2) {
    const int32_t tb = t + 1 < nt ? t + 1 : -1;
    tile_runs(plan, t, block_keys, lists[0]);
    tile_runs(plan, tb, block_keys, lists[1]);
    const int32_t begin = int32_t(plan.pblk.size() / 8);
    const int32_t n = merge_runs(lists, block_keys, plan.pblk);
    plan.pairs.insert(plan.pairs.end(), {t, tb, begin, n});
  }
}

// Work items of the paired-SM forward.  A couple is two consecutive tiles of
// one segment (offsets 2i and 2i + 1, or a segment's last odd tile alone):
// their key-block lists are the same up to one block, so one M = 256 product
// over a pair of SMs (one tile per SM) wastes almost nothing.  Couples are
// taken in the order their first tiles appear in the schedule (couple i of
// sibling segments side by side) and grouped two by two into quads: couple
// 2q in slot a, couple 2q + 1 in slot b.  A quad's merged block runs feed all
// four tiles (run slots a0, a1, b0, b1).
void build_quads(sp_plan &plan, int32_t block_keys) {
  plan.quads.clear();
  plan.qblk.clear();
  const int32_t nt = plan.n_tiles(), ns = plan.num_segments, tt = plan.tile_tokens;
  if (nt == 0) return;
  std::vector<int32_t> first(ns, INT32_MAX), count(ns, 0);
  for (int32_t t = 0; t < nt; ++t) {
    const int32_t sg = plan.tiles[5 * size_t(t)];
    first[sg] = std::min(first[sg], plan.tiles[5 * size_t(t) + 1]);
    ++count[sg];
  }
  std::vector<int64_t> base(size_t(ns) + 1, 0);
  for (int32_t sg = 0; sg < ns; ++sg) base[sg + 1] = base[sg] + count[sg];
  std::vector<int32_t> at(nt, -1);
  auto offset_of = [&](int32_t t) {
    return (plan.tiles[5 * size_t(t) + 1] - first[plan.tiles[5 * size_t(t)]]) / tt;
  };
  for (int32_t t = 0; t < nt; ++t) at[base[plan.tiles[5 * size_t(t)]] + offset_of(t)] = t;
  std::vector<int32_t> couples;  // [c][2]
  couples.reserve(size_t(nt) + 2);
  for (int32_t t = 0; t < nt; ++t) {
    const int32_t k = offset_of(t), sg = plan.tiles[5 * size_t(t)];
    if (k & 1) continue;
    couples.push_back(t);
    couples.push_back(k + 1 < count[sg] ? at[base[sg] + k + 1] : -1);
  }
  const int32_t nc = int32_t(couples.size() / 2);
  std::vector<TileRun> lists[4];
  for (int32_t c = 0; c < nc; c += 2) {
    const int32_t tiles4[4] = {couples[2 * size_t(c)], couples[2 * size_t(c) + 1],
                               c + 1 < nc ? couples[2 * size_t(c) + 2] : -1,
                               c + 1 < nc ? couples[2 * size_t(c) + 3] : -1};
    for (int i = 0; i < 4; ++i) tile_runs(plan, tiles4[i], block_keys, lists[i]);
    const int32_t begin = int32_t(plan.qblk.size() / 8);
    const int32_t n = merge_runs(lists, block_keys, plan.qblk);
    plan.quads.insert(plan.quads.end(), {tiles4[0], tiles4[1], tiles4[2], tiles4[3], begin, n});
  }
}

// Launch order of the backward's key blocks.  Each CTA re-reads Q and dO along
// its block's query run and adds dQ partials there, so CTAs that run at the
// same time should walk the same rows: blocks whose runs end at the same token
// (the same subtree end) are launched together and walk from that end in step.
// Within a group the longest run goes first.
void build_bwd_schedule(sp_plan &plan) {
  const int32_t n = plan.n_bwd();
  const int32_t *b = plan.bwd.data();
  std::vector<int32_t> idx(n);
  std::iota(idx.begin(), idx.end(), 0);
  auto len = [&](int32_t i) { return b[5 * i + 4] - b[5 * i + 3]; };
  std::stable_sort(idx.begin(), idx.end(), [&](int32_t x, int32_t y) {
    if (b[5 * x + 4] != b[5 * y + 4]) return b[5 * x + 4] > b[5 * y + 4];
    return len(x) > len(y);
  });
  plan.bwd_sched.clear();
  plan.bwd_run_sum = 0;
  plan.bwd_run_max = 0;
  for (int32_t i : idx) {
    plan.bwd_sched.insert(plan.bwd_sched.end(), b + 5 * i, b + 5 * i + 5);
    plan.bwd_run_sum += len(i);
    plan.bwd_run_max = std::max(plan.bwd_run_max, len(i));
  }
  build_bwd_merged(plan);
}

// Key blocks of the tensor-core backward.  A segment's last block is usually
// partial, yet it walks the segment's whole query run with all kv_block rows.
// Walking the keys in token order, such a block takes in the leading keys of
// the segments that follow it while they lie in its segment's subtree (their
// run end is at most the block's), so rows that would compute nothing work on
// the same query run; a segment whose leading keys were taken has its
// remaining keys blocked from there on.  The block's run is still
// [first key, subtree end of its first key's segment), and every key keeps
// its own run end in key_end, which the kernels mask with.  Rows {seg of the
// first key, first key, end key, first key, run end}, in the launch order of
// bwd_sched.
void build_bwd_merged(sp_plan &plan) {
  const int32_t n = plan.n_bwd(), B = plan.kv_block, T = plan.total_tokens;
  const int32_t *b = plan.bwd.data();
  plan.key_end.assign(size_t(std::max(T, 0)), 0);
  for (int32_t i = 0; i < n; ++i)
    for (int32_t k = b[5 * i + 1]; k < b[5 * i + 2]; ++k) plan.key_end[size_t(k)] = b[5 * i + 4];
  std::vector<int32_t> order(n);  // canonical rows by first key
  std::iota(order.begin(), order.end(), 0);
  std::sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return b[5 * x + 1] < b[5 * y + 1]; });
  std::vector<int32_t> from(n);  // first key of each row not yet placed
  for (int32_t i = 0; i < n; ++i) from[i] = b[5 * i + 1];
  std::vector<int32_t> rows;
  for (int32_t oi = 0; oi < n; ++oi) {
    const int32_t i = order[oi];
    const int32_t k0 = from[i], qe = b[5 * i + 4];
    int32_t k1 = b[5 * i + 2];
    if (k0 >= k1) continue;  // taken in whole by an earlier block
    for (int32_t oj = oi + 1; oj < n && k1 - k0 < B; ++oj) {
      const int32_t j = order[oj];
      if (from[j] != k1 || b[5 * j + 4] > qe) break;  // not contiguous, or outside the subtree
      const int32_t take = std::min(B - (k1 - k0), b[5 * j + 2] - from[j]);
      from[j] += take;
      k1 += take;
      if (from[j] < b[5 * j + 2]) break;
    }
    rows.insert(rows.end(), {b[5 * i], k0, k1, k0, qe});
  }
  const int32_t m = int32_t(rows.size() / 5);
  std::vector<int32_t> idx(m);
  std::iota(idx.begin(), idx.end(), 0);
  auto len = [&](int32_t i) { return rows[5 * size_t(i) + 4] - rows[5 * size_t(i) + 3]; };
  std::sort(idx.begin(), idx.end(), [&](int32_t x, int32_t y) {
    if (rows[5 * size_t(x) + 4] != rows[5 * size_t(y) + 4]) return rows[5 * size_t(x) + 4] > rows[5 * size_t(y) + 4];
    if (len(x) != len(y)) return len(x) > len(y);
    return rows[5 * size_t(x) + 1] < rows[5 * size_t(y) + 1];
  });
  plan.bwd_merged.clear();
  plan.bwdm_run_sum = 0;
  plan.bwdm_run_max = 0;
  for (int32_t i : idx) {
    plan.bwd_merged.insert(plan.bwd_merged.end(), rows.begin() + 5 * size_t(i), rows.begin() + 5 * size_t(i) + 5);
    plan.bwdm_run_sum += len(i);
    plan.bwdm_run_max = std::max(plan.bwdm_run_max, len(i));
  }
}

}  // namespace spc
