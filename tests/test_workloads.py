"""The seeded workloads match the recipe and the sizes stated for them.

A change to a generator would silently change every benchmarked workload and
parity case, so the documented figures are pinned here: token and segment
counts, leaves, depth, heads, edge-index counts, and the ranges the recipes
draw from.  CPU only; nothing here is the method's arithmetic.
"""
import numpy as np
import pytest
import torch

import workloads as W


def _stats(t):
    parent = np.asarray(t.parent)
    has_child = np.zeros(t.num_segments, dtype=bool)
    has_child[parent[parent >= 0]] = True
    kids = np.bincount(parent[parent >= 0], minlength=t.num_segments)
    return {"T": int(t.total_tokens), "segments": int(t.num_segments), "leaves": int((~has_child).sum()),
            "max_depth": int(np.max(t.depth)), "roots": int((parent == -1).sum()),
            "max_children": int(kids.max()), "children_of_internal": kids[has_child]}


@pytest.mark.parametrize("name,T,segments,leaves,max_depth,hq,hkv,D,edges", [
    ("tiny", 186, 6, 4, 2, 2, 2, 64, 8),
    ("star", 7659, 9, 8, 1, 32, 8, 128, 5611),
    ("forest", 323402, 272, 256, 1, 32, 8, 128, None),
    ("agent", 65536, 106, 58, 8, 32, 8, 128, 3419),
    ("long", 131072, 63, 28, 12, 64, 8, 128, None),
    ("forest_small", 40560, 34, 32, 1, 32, 8, 128, None),
    ("agent_small", 16384, 27, 13, 8, 32, 8, 128, 876),
    ("long_small", 16384, 16, 3, 12, 64, 8, 128, None),
])
def test_documented_sizes(name, T, segments, leaves, max_depth, hq, hkv, D, edges):
    w = W.get(name)
    s = _stats(w.tree)
    assert (s["T"], s["segments"], s["leaves"], s["max_depth"]) == (T, segments, leaves, max_depth)
    assert (w.hq, w.hkv, w.head_dim) == (hq, hkv, D)
    assert (None if w.edge_idx is None else len(w.edge_idx)) == edges
    assert w.softmax_scale == pytest.approx(1.0 / np.sqrt(D))


def test_recipe_ranges():
    star = W.grpo_star().tree
    assert int(star.seg_len[0]) == 2048 and all(256 <= int(x) <= 1024 for x in star.seg_len[1:])
    forest = W.grpo_forest().tree
    st = _stats(forest)
    assert st["roots"] == 16 and (st["children_of_internal"] == 16).all()
    roots = np.nonzero(np.asarray(forest.parent) == -1)[0]
    assert all(512 <= int(forest.seg_len[r]) <= 4096 for r in roots)
    assert all(128 <= int(forest.seg_len[s]) <= 2048 for s in range(forest.num_segments) if s not in set(roots))
    for name, lo, hi, kmax, dmax in (("agent", 16, 4096, 4, 8), ("long", 64, 8192, 3, 12)):
        t = W.get(name).tree
        st = _stats(t)
        assert st["max_children"] <= kmax and st["max_depth"] <= dmax
        # every segment's length is in the drawn range, except the one cut at the token cap
        out = [int(x) for x in t.seg_len[1:] if not lo <= int(x) <= hi]
        assert len(out) <= 1 and all(x < lo for x in out)
    assert int(W.long_fragment().tree.seg_len[0]) == 8192


def test_edge_indices_are_in_range_and_follow_the_recipe():
    tiny = W.tiny()
    leaf_tokens = set(np.arange(96, 186)) - set(np.arange(96, 144))  # leaves: seg1, seg3, seg4, seg5
    leaf_tokens |= set(np.arange(64, 96))
    assert len(set(tiny.edge_idx.tolist())) == 8 and set(tiny.edge_idx.tolist()) <= leaf_tokens
    star = W.grpo_star()
    assert np.array_equal(star.edge_idx, np.arange(2048, star.T))
    agent = W.agent_tree()
    assert agent.edge_idx.min() >= 0 and agent.edge_idx.max() < agent.T
    assert abs(len(agent.edge_idx) / agent.T - 0.05) < 0.005


def test_tensors_are_seeded_bf16_and_reproducible():
    w = W.tiny()
    a = W.draw_tensors(w, "bf16", with_hidden=True)
    b = W.draw_tensors(w, "bf16", with_hidden=True)
    for k in ("q", "k", "v", "do", "hidden"):
        assert a[k].dtype == torch.bfloat16 and torch.equal(a[k], b[k])
    assert tuple(a["q"].shape) == (186, 2, 64) and tuple(a["hidden"].shape) == (186, 256)
    lm = W.draw_lm_head(5, 64, 96, seed=3)
    assert tuple(lm["weight"].shape) == (96, 64) and int(lm["labels"].max()) < 96
