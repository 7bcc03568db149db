"""The planner tests catch planted mistakes in the library's host C++.

Each case plants one plausible mistake in a copy of ``plan.cpp`` (tree
validation, tiling, range merging, ordering, the backward table, the forward
pairs and quads and the backward launch order built at upload) or
``fragments.cpp`` (the bounded fragment planner).  The copy is built with g++
into a small host-only library, together with ``tests/c/planner_shim.cpp``.
The case then runs the checks the planner's parity tests make (hand-derived
plans, the oracle's planner and fragment planner on random trees, accepted and
refused trees) and expects at least one to fail.  No GPU, no CUDA.
"""
import shutil

import numpy as np
import pytest

import workloads as W
from oracle import fragments as OF
from oracle import plan as OP
from oracle import tree as OT

from host_planner import build_host_library, original_objects


pytestmark = pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")

# (file, text in it, replacement, what the mistake is)
MUTANTS = [
    ("plan.cpp", "merges[s] = p >= 0 && t.seg_start[p] + t.seg_len[p] == t.seg_start[s];", "merges[s] = false;",
     "touching ranges not merged"),
    ("plan.cpp", "merges[s] = p >= 0 && t.seg_start[p] + t.seg_len[p] == t.seg_start[s];",
     "merges[s] = p >= 0 && t.seg_start[p] == t.seg_start[s] - 1;", "merge test off by the parent's length"),
    ("plan.cpp", "if (t.seg_len[s] < 1 || t.seg_start[s] != pos)", "if (t.seg_len[s] < 0 || t.seg_start[s] != pos)",
     "empty segments accepted"),
    ("plan.cpp", "if (t.seg_len[s] < 1 || t.seg_start[s] != pos)", "if (t.seg_len[s] < 1 || t.seg_start[s] < pos)",
     "gaps accepted"),
    ("plan.cpp", "if (pos != t.total_tokens) return SP_ERR_INVALID_TREE;", "",
     "token total not checked"),
    ("plan.cpp", "(p < 0 ? 0 : t.depth[p] + 1)", "(p < 0 ? 0 : t.depth[p])", "depth not incremented"),
    ("plan.cpp", "while (!stack.empty() && stack.back() != p) stack.pop_back();",
     "if (!stack.empty() && stack.back() != p) stack.pop_back();", "preorder stack pops one level only"),
    ("plan.cpp", "if (stack.empty()) return SP_ERR_INVALID_TREE;", "",
     "closed parents accepted"),
    ("plan.cpp", "send[t.parent[s]] = std::max(send[t.parent[s]], send[s]);", "send[t.parent[s]] = send[s];",
     "subtree end from the first child only"),
    ("plan.cpp", "const int32_t q1 = std::min(a1, q0 + tile_tokens);", "const int32_t q1 = q0 + tile_tokens;",
     "tiles cross the segment end"),
    ("plan.cpp", "(int64_t(x.k) << 32) | x.seg,", "(int64_t(x.seg) << 32) | x.k,",
     "order 0 by segment before tile index (siblings not interleaved)"),
    ("plan.cpp", "{(int64_t(root[x.seg]) << 32) | int64_t(t.parent[x.seg] + 1),", "{int64_t(t.parent[x.seg] + 1),",
     "order 0 ignores the tree a tile belongs to"),
    ("plan.cpp", "keys[i] = {-x.kv_total,", "keys[i] = {x.kv_total,", "order 1 shortest first"),
    ("plan.cpp", "return x.a != y.a ? x.a < y.a : x.b < y.b;", "return x.a < y.a;", "ties of the first key left unordered"),
    ("plan.cpp", "if (cx != cy) return cx > cy;", "if (cx != cy) return cx < cy;", "backward table ascending"),
    ("plan.cpp", "blocks.push_back({s, k0, std::min(a1, k0 + kv_block), k0, send[s]});",
     "blocks.push_back({s, k0, std::min(a1, k0 + kv_block), a0, send[s]});",
     "block queries from the segment start"),
    ("plan.cpp", "const int32_t rb = int32_t(plan.ranges.size() / 2);",
     "const int32_t rb = int32_t(plan.ranges.size() / 2) - 1;", "range begin off by one"),
    ("plan.cpp", "      plan.ranges.back() = x.q1;\n    } else {\n      plan.ranges.push_back(a0);\n"
     "      plan.ranges.push_back(x.q1);",
     "      plan.ranges.back() = a0 + t.seg_len[x.seg];\n    } else {\n      plan.ranges.push_back(a0);\n"
     "      plan.ranges.push_back(a0 + t.seg_len[x.seg]);", "own range to the segment end"),
    ("plan.cpp", "int32_t(plan.ranges.size() / 2) > rb && plan.ranges.back() == a0",
     "int32_t(plan.ranges.size() / 2) > rb && false", "own range not merged into a touching parent range"),
    ("plan.cpp", "anc_tokens[s] = anc_tokens[p] + t.seg_len[p];", "anc_tokens[s] = t.seg_len[p];",
     "longest-first key counts the parent only"),
    ("plan.cpp", "e, r + 1 == tl[4]});", "e, r == 0});", "forward blocks flagged causal on the first range"),
    ("plan.cpp", "int32_t((int64_t(e) - a + block_keys - 1) / block_keys)", "int32_t((int64_t(e) - a) / block_keys)",
     "a range's partial last block dropped"),
    ("plan.cpp", "const int32_t tb = t + 1 < nt ? t + 1 : -1;", "const int32_t tb = t + 1 < nt ? t + 1 : t;",
     "an odd last tile paired with itself"),
    ("plan.cpp", "        n = std::min(n, (c - kb + block_keys - 1) / block_keys);  // stop before tile i's next block\n",
     "", "a run not stopped where another tile's block starts"),
    ("plan.cpp", "flags |= tr.causal ? (1 << i) : 0;", "flags |= tr.causal ? (1 << (i & 1)) : 0;",
     "causal bits of slots 2 and 3 written to slots 0 and 1"),
    ("plan.cpp", "if (e[i] != 0 && (bi[i] += n) == lists[i][ri[i]].nb) {", "if (e[i] != 0 && (bi[i] += 1) == lists[i][ri[i]].nb) {",
     "a merged run advances its tiles by one block"),
    ("plan.cpp", "return b[5 * x + 4] > b[5 * y + 4];", "return b[5 * x + 4] < b[5 * y + 4];",
     "backward launch order by earliest run end"),
    ("plan.cpp", "    return len(x) > len(y);", "    return len(x) < len(y);", "backward runs of one end shortest first"),
    ("plan.cpp", "plan.bwd_run_max = std::max(plan.bwd_run_max, len(i));", "plan.bwd_run_max = len(i);",
     "longest backward run mis-counted"),
    ("plan.cpp", "plan.bwd_run_sum += len(i);", "plan.bwd_run_sum = len(i);", "backward run sum mis-counted"),
    ("plan.cpp", "couples.push_back(k + 1 < count[sg] ? at[base[sg] + k + 1] : -1);",
     "couples.push_back(k + 2 < count[sg] ? at[base[sg] + k + 1] : -1);", "a segment's last partner tile dropped"),
    ("plan.cpp", "    if (k & 1) continue;", "    if (!(k & 1)) continue;", "couples started on odd tiles"),
    ("plan.cpp", "                               c + 1 < nc ? couples[2 * size_t(c) + 2] : -1,",
     "                               c + 1 < nc ? couples[2 * size_t(c)] : -1,", "a quad's slot b repeats slot a"),
    ("fragments.cpp", "if (!cur_seg.empty() && cur_tokens + extra > cap) {",
     "if (!cur_seg.empty() && cur_tokens + extra >= cap) {", "a fragment never fills the cap exactly"),
    ("fragments.cpp", "      emit();\n      extra = path_tokens;", "      emit();",
     "a new fragment's tokens miss the re-added ancestors"),
    ("fragments.cpp", "cur_owned.push_back(*it == s ? 1 : 0);", "cur_owned.push_back(1);",
     "re-added ancestors owned again"),
    ("fragments.cpp", "f.local_parent.push_back(t.parent[s] >= 0 ? local[t.parent[s]] : -1);",
     "f.local_parent.push_back(t.parent[s]);", "local parent is the whole tree's parent"),
    ("fragments.cpp", "      f.local_start.push_back(start);\n      start += t.seg_len[s];",
     "      start += t.seg_len[s];\n      f.local_start.push_back(start);", "local starts shifted by a segment"),
    ("fragments.cpp", "if (path_tokens > cap) return SP_ERR_CAP;", "if (path_tokens >= cap) return SP_ERR_CAP;",
     "a root path exactly at the cap refused"),
    ("fragments.cpp", "      local[s] = -1;\n      in_cur[s] = 0;", "      local[s] = -1;",
     "segments of a closed fragment still counted as present"),
]


def _expected_fragment_tables(t, frags):
    seg, owned, lpar, lstart, offsets, tokens = [], [], [], [], [0], []
    for f in frags:
        local, start = {}, 0
        for a, o in f:
            local[a] = len(local)
            seg.append(a)
            owned.append(int(o))
            lpar.append(local[int(t.parent[a])] if int(t.parent[a]) >= 0 else -1)
            lstart.append(start)
            start += int(t.seg_len[a])
        offsets.append(offsets[-1] + len(f))
        tokens.append(start)
    return {"seg": seg, "owned": owned, "local_parent": lpar, "local_start": lstart, "offsets": offsets,
            "tokens": tokens}


def _battery(host):
    """The planner's parity checks against one build; raises AssertionError at the first difference."""
    from test_oracle import FOREST_HAND, _read_golden
    gold = _read_golden()

    class Ok:
        """The build's calls on valid input: a refusal is a failed check."""

        @staticmethod
        def plan(*a, **k):
            r = host.plan(*a, **k)
            assert not isinstance(r, int), f"a valid tree was refused (status {r})"
            return r

        @staticmethod
        def device_tables(*a):
            r = host.device_tables(*a)
            assert not isinstance(r, int), f"a valid tree was refused (status {r})"
            return r

        @staticmethod
        def fragments(*a):
            r = host.fragments(*a)
            assert not isinstance(r, int), f"a feasible fragment plan was refused (status {r})"
            return r

    t = W.tiny().tree
    args = (t.seg_start, t.seg_len, t.parent, t.depth)
    tiles, ranges, bwd = Ok.plan(*args, 32, 32, 0)
    got = [(int(s), int(a), int(b), [tuple(map(int, ranges[r])) for r in range(rb, rb + rc)])
           for s, a, b, rb, rc in tiles]
    assert got == gold["tiles"]
    assert [tuple(map(int, b)) for b in bwd] == gold["bwd"]
    tiles1 = Ok.plan(*args, 32, 32, 1)[0]
    assert [tuple(map(int, r[:3])) for r in tiles1] == gold["order1"]
    f = FOREST_HAND
    tiles, ranges, bwd = Ok.plan(f["seg_start"], f["seg_len"], f["parent"], f["depth"], 32, 32, 0)
    assert [(int(s), int(a), int(b), [tuple(map(int, ranges[r])) for r in range(rb, rb + rc)])
            for s, a, b, rb, rc in tiles] == f["tiles"]
    # refused trees (and a wrong token total); every one must come back as an invalid tree
    base = [np.asarray(a).copy() for a in args]
    bad = []
    for i, pos, val in ((1, 2, 0), (0, 3, 150), (2, 1, 3), (3, 3, 1), (2, 4, -2)):
        a = [x.copy() for x in base]
        a[i][pos] = val
        bad.append((a, None))
    a = [x.copy() for x in base]
    a[2][5], a[3][5] = 1, 2  # not preorder
    bad.append((a, None))
    a = [x.copy() for x in base]
    a[1][4], a[0][5] = 0, 160  # empty segment, consistent packing
    bad.append((a, None))
    bad.append(([x.copy() for x in base], 187))  # wrong total
    for a, total in bad:
        assert host.plan(*a, 32, 32, 0, total=total) == -1
    assert host.fragments(*args, 127) == -10
    # the tables the kernels read, as the first upload builds them
    from test_device_tables import check_device_tables
    for name in ("tiny", "star"):
        w = W.get(name)
        wt = w.tree
        check_device_tables(w.T, Ok.device_tables(wt.seg_start, wt.seg_len, wt.parent, wt.depth,
                                                  128 // (w.hq // w.hkv), 128, 0))
    # the run merge on lists whose ranges start at keys that do not line up (a run must stop where
    # another slot's next block starts); the plans above never produce such lists
    from test_device_tables import check_run_merge, random_run_lists
    rng_t = np.random.default_rng(17)
    for _ in range(60):
        check_run_merge(host, random_run_lists(rng_t))
    rng = np.random.default_rng(5)
    for _ in range(40):
        r = W.random_small_tree(rng, max_segments=12, max_len=30)
        ra = (r.seg_start, r.seg_len, r.parent, r.depth)
        tt, kb, order = int(rng.integers(1, 33)), int(rng.integers(1, 33)), int(rng.integers(0, 2))
        for g, w in zip(Ok.plan(*ra, tt, kb, order), OP.build(r.seg_start, r.seg_len, r.parent, tt, kb, order)):
            assert np.array_equal(g, w)
        lp = max(sum(int(r.seg_len[x]) for x in OT.ancestors(r.parent, s) + [s]) for s in range(r.num_segments))
        for cap in (lp, int(rng.integers(lp, 3 * lp + 1))):
            got = Ok.fragments(*ra, cap)
            want = _expected_fragment_tables(r, OF.plan_fragments(r.seg_len, r.parent, cap))
            for k, v in want.items():
                assert list(got[k]) == v, k


@pytest.fixture(scope="module")
def objects(tmp_path_factory):
    d = tmp_path_factory.mktemp("host_mutants")
    return d, original_objects(d)


def test_unmutated_host_code_passes_the_battery(objects):
    d, objs = objects
    _battery(build_host_library(objs, d / "original"))


@pytest.mark.parametrize("mutant", MUTANTS, ids=[f"{m[0]}: {m[3]}" for m in MUTANTS])
def test_planted_host_mistake_is_caught(objects, mutant):
    d, objs = objects
    host = build_host_library(objs, d / f"m{MUTANTS.index(mutant)}", mutant)
    with pytest.raises(AssertionError):
        _battery(host)
