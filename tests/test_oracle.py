"""Pins for the CPU oracle: brute force, library routines, finite differences,
closed forms and invariants.  Nothing here touches the CUDA library."""
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from oracle import gather as OG
from oracle import plan as OP
from oracle import tree as OT

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, T, hq, hkv, D, scale=1.0):
    q = rng.standard_normal((T, hq, D)) * scale
    k = rng.standard_normal((T, hkv, D)) * scale
    v = rng.standard_normal((T, hkv, D)) * scale
    do = rng.standard_normal((T, hq, D))
    return q, k, v, do


def _sdpa_causal(q, k, v, scale):
    """torch's own causal attention in fp64 on [T, H, D] arrays (GQA expanded)."""
    G = q.shape[1] // k.shape[1]
    qt = torch.tensor(q).permute(1, 0, 2)[None]
    kt = torch.tensor(k).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    vt = torch.tensor(v).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def _tree_args(t):
    return t.seg_start, t.seg_len, t.parent


# ---------------------------------------------------------------- tree checks

def test_validate_accepts_generated_configs():
    for name in ("tiny", "star", "agent", "long"):
        t = W.get(name).tree
        OT.validate(t.seg_start, t.seg_len, t.parent, t.depth, t.total_tokens)


@pytest.mark.parametrize("mutate,msg", [
    (lambda a: a["seg_len"].__setitem__(2, 0), "empty"),
    (lambda a: a["seg_start"].__setitem__(3, 100), "start"),
    (lambda a: a["seg_start"].__setitem__(3, 150), "gap"),
    (lambda a: a["parent"].__setitem__(1, 3), "parent"),
    (lambda a: a["parent"].__setitem__(0, 0), "root"),
    (lambda a: a["depth"].__setitem__(3, 1), "depth"),
    (lambda a: (a["parent"].__setitem__(5, 1), a["depth"].__setitem__(5, 2)), "preorder"),
])
def test_validate_rejects(mutate, msg):
    t = W.tiny().tree
    a = {k: getattr(t, k).copy() for k in ("seg_start", "seg_len", "parent", "depth")}
    mutate(a)
    with pytest.raises(OT.InvalidTree):
        OT.validate(a["seg_start"], a["seg_len"], a["parent"], a["depth"], t.total_tokens)


def test_validate_rejects_an_empty_segment_even_when_the_packing_is_consistent():
    # the tiny tree with leaf segment 4 emptied and every later start moved back to stay packed
    with pytest.raises(OT.InvalidTree):
        OT.validate([0, 64, 96, 144, 160, 160], [64, 32, 48, 16, 0, 17], [-1, 0, 0, 2, 2, 0],
                    [0, 1, 1, 2, 2, 1], 177)


def test_visibility_pairs_and_naive_tokens_match_hand_count():
    gold = _read_golden()
    t = W.tiny().tree
    m = OT.visible_mask_bruteforce(*_tree_args(t))
    assert int(m.sum()) == gold["pairs"]
    naive = sum(len(OT.path_tokens(t.seg_start, t.seg_len, t.parent, l)) for l in OT.leaves(t.parent))
    assert naive == gold["naive_tokens"]


# ---------------------------------------------------------------- plan checks

def _read_golden():
    tiles, bwd, order1, out = [], [], [], {}
    with open(os.path.join(GOLDEN, "tiny_plan.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            if line.startswith("tile "):
                head, rng = line[5:].split("|")
                s, q0, q1 = map(int, head.split())
                r = list(map(int, rng.split()))
                tiles.append((s, q0, q1, list(zip(r[0::2], r[1::2]))))
            elif line.startswith("bwd "):
                bwd.append(tuple(map(int, line[4:].split())))
            elif line.startswith("order1 "):
                order1.append(tuple(map(int, line[7:].split())))
            else:
                k, v = line.split()
                out[k] = int(v)
    out["tiles"], out["bwd"], out["order1"] = tiles, bwd, order1
    return out


def test_plan_matches_hand_derived_golden():
    gold = _read_golden()
    t = W.tiny().tree
    tiles, ranges, bwd = OP.build(*_tree_args(t), tile_tokens=32, kv_block=32, order=0)
    got = [(int(s), int(q0), int(q1), [tuple(map(int, ranges[r])) for r in range(rb, rb + rc)])
           for s, q0, q1, rb, rc in tiles]
    assert got == gold["tiles"]
    assert [tuple(map(int, b)) for b in bwd] == gold["bwd"]
    # r_begin is the running count of ranges in schedule order
    assert list(tiles[:, 3]) == list(np.cumsum([0] + [len(x[3]) for x in gold["tiles"]])[:-1])


def test_plan_order1_matches_hand_derived_golden():
    gold = _read_golden()
    t = W.tiny().tree
    tiles, _, _ = OP.build(*_tree_args(t), tile_tokens=32, kv_block=32, order=1)
    assert [tuple(map(int, r[:3])) for r in tiles] == gold["order1"]


# Two trees: root 0 [0,40) with children 1 [40,60) and 2 [60,80); root 3 [80,110) with child 4
# [110,120).  Tiles of 32 tokens in order 0, worked by hand: the first tree's tiles, then the
# second's; each tile's ranges are its ancestors' tokens and its own segment up to the tile end.
FOREST_HAND = {
    "seg_start": [0, 40, 60, 80, 110], "seg_len": [40, 20, 20, 30, 10], "parent": [-1, 0, 0, -1, 3],
    "depth": [0, 1, 1, 0, 1],
    "tiles": [(0, 0, 32, [(0, 32)]), (0, 32, 40, [(0, 40)]), (1, 40, 60, [(0, 60)]),
              (2, 60, 80, [(0, 40), (60, 80)]), (3, 80, 110, [(80, 110)]), (4, 110, 120, [(80, 120)])],
    # kv_block 32: (seg, kv_start, kv_end, q_begin, q_end), most queries first, ties by kv_start
    "bwd": [(0, 0, 32, 0, 80), (0, 32, 40, 32, 80), (3, 80, 110, 80, 120), (1, 40, 60, 40, 60),
            (2, 60, 80, 60, 80), (4, 110, 120, 110, 120)],
}


def test_plan_forest_keeps_each_tree_together_by_hand():
    f = FOREST_HAND
    tiles, ranges, bwd = OP.build(f["seg_start"], f["seg_len"], f["parent"], tile_tokens=32, kv_block=32,
                                  order=0)
    got = [(int(s), int(q0), int(q1), [tuple(map(int, ranges[r])) for r in range(rb, rb + rc)])
           for s, q0, q1, rb, rc in tiles]
    assert got == f["tiles"]
    assert [tuple(map(int, b)) for b in bwd] == f["bwd"]


def test_plan_order0_groups_tiles_by_tree_on_the_forest_workload():
    t = W.grpo_forest().tree
    tiles, _, _ = OP.build(*_tree_args(t), tile_tokens=32, kv_block=128, order=0)
    root = np.empty(t.num_segments, dtype=np.int64)
    for s in range(t.num_segments):
        root[s] = s if t.parent[s] == -1 else root[t.parent[s]]
    seq = root[tiles[:, 0]]
    assert (np.diff(seq) >= 0).all() and len(np.unique(seq)) == int((np.asarray(t.parent) == -1).sum()) > 1


@pytest.mark.parametrize("seed", range(200))
def test_plan_masks_equal_bruteforce(seed):
    rng = np.random.default_rng(1000 + seed)
    t = W.random_small_tree(rng, max_segments=7, max_len=12)
    T = t.total_tokens
    brute = OT.visible_mask_bruteforce(*_tree_args(t))
    tt = int(rng.integers(1, 9))
    kb = int(rng.integers(1, 9))
    for order in (0, 1):
        tiles, ranges, bwd = OP.build(*_tree_args(t), tile_tokens=tt, kv_block=kb, order=order)
        assert np.array_equal(OP.expand_forward_mask(T, tiles, ranges), brute)
        assert np.array_equal(OP.expand_backward_mask(T, bwd), brute)
        # every query token in exactly one tile, every key in exactly one block
        cover = np.zeros(T, int)
        for s, q0, q1, rb, rc in tiles:
            cover[q0:q1] += 1
        assert (cover == 1).all()
        cover[:] = 0
        for s, k0, k1, q0, q1 in bwd:
            cover[k0:k1] += 1
        assert (cover == 1).all()
    # closed form: j visible to i  <=>  j <= i < end of seg(j)'s subtree
    seg = OT.segment_of_token(t.seg_start, t.seg_len)
    send = np.array([OP.subtree_end(*_tree_args(t), s) for s in range(t.num_segments)])
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    assert np.array_equal((j <= i) & (i < send[seg][None, :]), brute)


def test_plan_order_keeps_siblings_adjacent():
    t = W.grpo_star().tree
    tiles, _, _ = OP.build(*_tree_args(t), tile_tokens=32, kv_block=128, order=0)
    # after the prompt's tiles, tile k of all 8 completions run back to back
    first = [int(s) for s in tiles[64:72, 0]]
    assert first == list(range(1, 9))


# ---------------------------------------------------------- attention: pins

def test_single_segment_equals_library_causal_attention():
    rng = np.random.default_rng(7)
    q, k, v, do = _rand(rng, 97, 4, 2, 16)
    seg_start, seg_len, parent = [0], [97], [-1]
    O, LSE = A.tree_forward(q, k, v, seg_start, seg_len, parent, 0.25)
    np.testing.assert_allclose(O, _sdpa_causal(q, k, v, 0.25), rtol=0, atol=1e-12)
    # gradients against torch autograd through the same library routine
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = 2
    o = torch.nn.functional.scaled_dot_product_attention(
        tq.permute(1, 0, 2)[None], tk.repeat_interleave(G, 1).permute(1, 0, 2)[None],
        tv.repeat_interleave(G, 1).permute(1, 0, 2)[None], is_causal=True, scale=0.25)
    (o[0].permute(1, 0, 2) * torch.tensor(do)).sum().backward()
    dQ, dK, dV = A.tree_backward(q, k, v, do, seg_start, seg_len, parent, 0.25)
    for ours, ref in ((dQ, tq.grad), (dK, tk.grad), (dV, tv.grad)):
        np.testing.assert_allclose(ours, ref.numpy(), rtol=0, atol=1e-11)


def test_large_scores_stay_finite_and_match_the_library():
    """Scores of several hundred (far beyond exp's range in fp64) through both routes and the backward."""
    rng = np.random.default_rng(18)
    q, k, v, do = _rand(rng, 60, 2, 1, 16, scale=30.0)
    ref = _sdpa_causal(q, k, v, 0.25)
    mask = np.tril(np.ones((60, 60), dtype=bool))
    assert np.abs(0.25 * np.einsum("id,jd->ij", q[:, 0], k[:, 0])).max() > 800
    O, L = A.tree_forward(q, k, v, [0], [60], [-1], 0.25)
    O2, L2, _ = A.dense_forward(q, k, v, mask, 0.25)
    for o, l in ((O, L), (O2, L2)):
        assert np.isfinite(o).all() and np.isfinite(l).all()
        np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-10)
    for g in A.tree_backward(q, k, v, do, [0], [60], [-1], 0.25) + A.dense_backward(q, k, v, do, mask, 0.25):
        assert np.isfinite(g).all()


def test_star_with_one_child_equals_causal_on_concatenation():
    rng = np.random.default_rng(8)
    q, k, v, _ = _rand(rng, 50, 2, 2, 8)
    O, _ = A.tree_forward(q, k, v, [0, 30], [30, 20], [-1, 0], 0.5)
    np.testing.assert_allclose(O, _sdpa_causal(q, k, v, 0.5), rtol=0, atol=1e-12)


def test_lse_is_log_sum_exp_over_visible_keys():
    t = W.tiny().tree
    rng = np.random.default_rng(9)
    q, k, v, _ = _rand(rng, t.total_tokens, 2, 1, 8)
    _, LSE = A.tree_forward(q, k, v, *_tree_args(t), 0.3)
    m = OT.visible_mask_bruteforce(*_tree_args(t))
    for h in range(2):
        for i in range(0, t.total_tokens, 7):
            js = np.nonzero(m[i])[0]
            s = [0.3 * float(np.dot(q[i, h], k[j, 0])) for j in js]
            assert abs(LSE[h, i] - np.log(np.sum(np.exp(s)))) < 1e-12


@pytest.mark.parametrize("seed", range(50))
def test_unrolled_equals_dense_tree_mask(seed):
    rng = np.random.default_rng(seed)
    t = W.random_small_tree(rng, max_segments=7, max_len=20)
    hkv = int(rng.integers(1, 3))
    hq = hkv * int(rng.choice([1, 2]))
    q, k, v, do = _rand(rng, t.total_tokens, hq, hkv, 8)
    mask = OT.visible_mask_bruteforce(*_tree_args(t))
    O1, L1 = A.tree_forward(q, k, v, *_tree_args(t), 0.4)
    O2, L2, _ = A.dense_forward(q, k, v, mask, 0.4)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L1, L2, rtol=0, atol=1e-12)
    g1 = A.tree_backward(q, k, v, do, *_tree_args(t), 0.4)
    g2 = A.dense_backward(q, k, v, do, mask, 0.4)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


def test_dense_route_matches_library_masked_attention_and_autograd():
    t = W.tiny().tree
    rng = np.random.default_rng(11)
    q, k, v, do = _rand(rng, t.total_tokens, 2, 2, 8)
    mask = OT.visible_mask_bruteforce(*_tree_args(t))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(
        tq.permute(1, 0, 2)[None], tk.permute(1, 0, 2)[None], tv.permute(1, 0, 2)[None],
        attn_mask=torch.tensor(mask), scale=0.35)
    (o[0].permute(1, 0, 2) * torch.tensor(do)).sum().backward()
    O, _, _ = A.dense_forward(q, k, v, mask, 0.35)
    np.testing.assert_allclose(O, o[0].permute(1, 0, 2).detach().numpy(), rtol=0, atol=1e-12)
    dQ, dK, dV = A.dense_backward(q, k, v, do, mask, 0.35)
    for ours, ref in ((dQ, tq.grad), (dK, tk.grad), (dV, tv.grad)):
        np.testing.assert_allclose(ours, ref.numpy(), rtol=0, atol=1e-11)


def test_softmax_rows_sum_to_one_over_visible_keys_only():
    t = W.tiny().tree
    rng = np.random.default_rng(19)
    q, k, v, _ = _rand(rng, t.total_tokens, 2, 1, 8)
    mask = OT.visible_mask_bruteforce(*_tree_args(t))
    _, _, P = A.dense_forward(q, k, v, mask, 0.4)
    np.testing.assert_allclose(P.sum(axis=2), 1.0, rtol=0, atol=1e-13)
    assert (P[:, ~mask] == 0).all() and (P[:, mask] > 0).all()


def test_gradients_match_finite_differences():
    t = W.tiny().tree
    rng = np.random.default_rng(12)
    q, k, v, do = _rand(rng, t.total_tokens, 2, 1, 8, 0.7)
    args = _tree_args(t)
    scale = 0.35

    def loss(q_, k_, v_):
        O, _ = A.tree_forward(q_, k_, v_, *args, scale)
        return float((O * do).sum())

    dQ, dK, dV = A.tree_backward(q, k, v, do, *args, scale)
    h = 1e-6
    for trial in range(32):  # random directions
        u = [rng.standard_normal(x.shape) for x in (q, k, v)]
        fp = loss(q + h * u[0], k + h * u[1], v + h * u[2])
        fm = loss(q - h * u[0], k - h * u[1], v - h * u[2])
        fd = (fp - fm) / (2 * h)
        an = float((dQ * u[0]).sum() + (dK * u[1]).sum() + (dV * u[2]).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an))
    # single coordinates: each (tensor, entry) in isolation
    for trial in range(200):
        which = trial % 3
        x = [q, k, v][which]
        pos = tuple(int(rng.integers(0, n)) for n in x.shape)
        e = np.zeros_like(x)
        e[pos] = 1.0
        xs = [q, k, v]
        p = [a + h * e if i == which else a for i, a in enumerate(xs)]
        m = [a - h * e if i == which else a for i, a in enumerate(xs)]
        fd = (loss(*p) - loss(*m)) / (2 * h)
        an = [dQ, dK, dV][which][pos]
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an))


def test_loss_owner_choice_does_not_change_gradients():
    t = W.tiny().tree
    rng = np.random.default_rng(13)
    q, k, v, do = _rand(rng, t.total_tokens, 2, 2, 8)
    g1 = A.tree_backward(q, k, v, do, *_tree_args(t), 0.4, owner="first")
    g2 = A.tree_backward(q, k, v, do, *_tree_args(t), 0.4, owner="last")
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_gradient_sums():
    """sum_j dV_j = sum_i dO_i (rows of P sum to 1); sum_j dK_j = 0 (rows of dS sum to 0)."""
    t = W.tiny().tree
    rng = np.random.default_rng(14)
    q, k, v, do = _rand(rng, t.total_tokens, 4, 2, 8)
    dQ, dK, dV = A.tree_backward(q, k, v, do, *_tree_args(t), 0.4)
    for g in range(2):
        np.testing.assert_allclose(dV[:, g].sum(0), do[:, 2 * g:2 * g + 2].sum((0, 1)), atol=1e-11)
        np.testing.assert_allclose(dK[:, g].sum(0), 0.0, atol=1e-11)


def _permute_siblings(t, rng):
    """Re-lay the tree with every node's children in a random order.

    Returns the new tree and new_index_of_old_token."""
    ch = OT.children(t.parent)
    roots = [s for s in range(t.num_segments) if t.parent[s] == -1]
    order, pars = [], []
    newid = {}

    def visit(s, p):
        newid[s] = len(order)
        order.append(s)
        pars.append(p)
        kids = list(ch[s])
        rng.shuffle(kids)
        for c in kids:
            visit(c, newid[s])

    for r in roots:
        visit(r, -1)
    nt = W.tree_from_preorder([int(t.seg_len[s]) for s in order], pars)
    perm = np.empty(t.total_tokens, dtype=np.int64)
    for s in order:
        a = int(t.seg_start[s])
        b = int(nt.seg_start[newid[s]])
        perm[a:a + int(t.seg_len[s])] = np.arange(b, b + int(t.seg_len[s]))
    return nt, perm


def test_sibling_permutation_leaves_results_unchanged():
    t = W.tiny().tree
    rng = np.random.default_rng(15)
    q, k, v, do = _rand(rng, t.total_tokens, 2, 1, 8)
    O, L = A.tree_forward(q, k, v, *_tree_args(t), 0.4)
    g = A.tree_backward(q, k, v, do, *_tree_args(t), 0.4)
    for trial in range(4):
        nt, perm = _permute_siblings(t, rng)
        inv = np.argsort(perm)
        q2, k2, v2, do2 = (x[inv] for x in (q, k, v, do))
        O2, L2 = A.tree_forward(q2, k2, v2, *_tree_args(nt), 0.4)
        np.testing.assert_allclose(O2[perm], O, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L2[:, perm], L, rtol=0, atol=1e-12)
        g2 = A.tree_backward(q2, k2, v2, do2, *_tree_args(nt), 0.4)
        for a, b in zip(g2, g):
            np.testing.assert_allclose(a[perm], b, rtol=0, atol=1e-12)


def test_sibling_isolation():
    """Changing one branch's K/V changes nothing outside that branch's subtree."""
    t = W.tiny().tree
    rng = np.random.default_rng(16)
    q, k, v, _ = _rand(rng, t.total_tokens, 2, 1, 8)
    O, L = A.tree_forward(q, k, v, *_tree_args(t), 0.4)
    k2, v2 = k.copy(), v.copy()
    k2[96:169] += 1.0  # seg2 and its subtree (seg3, seg4)
    v2[96:169] -= 2.0
    O2, L2 = A.tree_forward(q, k2, v2, *_tree_args(t), 0.4)
    outside = np.r_[0:96, 169:186]
    assert np.array_equal(O2[outside], O[outside])
    assert np.array_equal(L2[:, outside], L[:, outside])
    assert not np.allclose(O2[96:169], O[96:169])


def test_bf16_inputs_are_upcast_exactly():
    w = W.tiny()
    x = W.draw_tensors(w, "bf16")
    q = x["q"].float().numpy()
    assert np.array_equal(q.astype(np.float64), x["q"].double().numpy())


def test_edge_gather_oracle():
    h = np.arange(12.0).reshape(6, 2)
    out = OG.edge_gather(h, [5, 0, 5])
    assert out.tolist() == [[10.0, 11.0], [0.0, 1.0], [10.0, 11.0]]
    assert OG.edge_gather(h, []).shape == (0, 2)
    with pytest.raises(IndexError):
        OG.edge_gather(h, [6])
    with pytest.raises(IndexError):
        OG.edge_gather(h, [-1])
    for bad in ([6], [-1], [0, -1]):
        with pytest.raises(IndexError):
            OG.edge_gather_backward(np.ones((len(bad), 2)), bad, 6)


def test_subtree_key_grads_equal_full_backward():
    t = W.tiny().tree
    rng = np.random.default_rng(17)
    q, k, v, do = _rand(rng, t.total_tokens, 4, 2, 8)
    _, dK, dV = A.tree_backward(q, k, v, do, *_tree_args(t), 0.4)
    for s in range(t.num_segments):
        a0, a1 = int(t.seg_start[s]), int(t.seg_start[s] + t.seg_len[s])
        for g in range(2):
            sk, sv = A.subtree_key_grads(q, k, v, do, *_tree_args(t), 0.4, s, g)
            np.testing.assert_allclose(sk, dK[a0:a1, g], rtol=0, atol=1e-12)
            np.testing.assert_allclose(sv, dV[a0:a1, g], rtol=0, atol=1e-12)


def test_edge_gather_backward_is_the_adjoint_of_the_gather():
    """<gather(h), g> == <h, gather_backward(g)> for random h, g (duplicates included)."""
    rng = np.random.default_rng(31)
    T, Hd = 40, 6
    idx = np.concatenate([rng.integers(0, T, 25), [3, 3, 3, 17]])
    h = rng.standard_normal((T, Hd))
    g = rng.standard_normal((len(idx), Hd))
    lhs = float((OG.edge_gather(h, idx) * g).sum())
    rhs = float((h * OG.edge_gather_backward(g, idx, T)).sum())
    assert abs(lhs - rhs) < 1e-12
    gb = OG.edge_gather_backward(g, idx, T)
    assert np.array_equal(gb[3], g[np.nonzero(idx == 3)[0]].sum(0))
    untouched = np.setdiff1d(np.arange(T), idx)
    assert (gb[untouched] == 0).all()


# ------------------------------------------------------------ vocabulary head (log-probabilities)

def _lmh_case(E=5, V=11, Hd=7, seed=0):
    r = np.random.default_rng(seed)
    return r.standard_normal((E, Hd)), r.standard_normal((V, Hd)) * 0.7, r.integers(0, V, E)


def test_lm_head_zero_weight_gives_uniform_distribution():
    from oracle import lm_head as LH
    h, w, y = _lmh_case()
    lp, lse = LH.edge_logprob(h, np.zeros_like(w), y)
    np.testing.assert_allclose(lp, -np.log(w.shape[0]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, np.log(w.shape[0]), rtol=0, atol=1e-15)


def test_lm_head_probabilities_sum_to_one_over_the_vocabulary():
    from oracle import lm_head as LH
    h, w, _ = _lmh_case(E=3, V=9)
    total = np.zeros(3)
    for v in range(9):
        lp, _ = LH.edge_logprob(h, w, np.full(3, v))
        total += np.exp(lp)
    np.testing.assert_allclose(total, 1.0, rtol=0, atol=1e-13)


def test_lm_head_matches_scipy_log_softmax():
    from scipy.special import log_softmax
    from oracle import lm_head as LH
    h, w, y = _lmh_case(E=6, V=13, Hd=5, seed=3)
    lp, _ = LH.edge_logprob(h, w, y)
    ref = log_softmax(np.einsum("ed,vd->ev", h, w), axis=1)[np.arange(6), y]
    np.testing.assert_allclose(lp, ref, rtol=0, atol=1e-12)


def test_lm_head_is_invariant_to_a_shift_shared_by_all_vocabulary_rows():
    from oracle import lm_head as LH
    h, w, y = _lmh_case(seed=4)
    a = np.random.default_rng(5).standard_normal(w.shape[1])
    lp0, lse0 = LH.edge_logprob(h, w, y)
    lp1, lse1 = LH.edge_logprob(h, w + a[None, :], y)
    np.testing.assert_allclose(lp1, lp0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse1 - lse0, h @ a, rtol=0, atol=1e-12)


def test_lm_head_does_not_overflow_on_large_logits():
    from oracle import lm_head as LH
    h = np.array([[1.0, 0.0]])
    w = np.array([[2000.0, 0.0], [0.0, 0.0], [1990.0, 0.0]])
    lp, lse = LH.edge_logprob(h, w, np.array([0]))
    assert np.isfinite(lp).all() and np.isfinite(lse).all()
    np.testing.assert_allclose(lp, -np.log1p(np.exp(-10.0) + np.exp(-2000.0)), rtol=0, atol=1e-12)


def test_lm_head_backward_matches_finite_differences():
    from oracle import lm_head as LH
    h, w, y = _lmh_case(E=3, V=5, Hd=4, seed=6)
    g = np.random.default_rng(7).standard_normal(3)
    dh, dw = LH.edge_logprob_backward(h, w, y, g)
    loss = lambda hh, ww: float(np.dot(g, LH.edge_logprob(hh, ww, y)[0]))
    eps = 1e-6
    for arr, grad, which in ((h, dh, 0), (w, dw, 1)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            lp_ = loss(p, w) if which == 0 else loss(h, p)
            lm_ = loss(m, w) if which == 0 else loss(h, m)
            num[idx] = (lp_ - lm_) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=0, atol=1e-7)


def test_lm_head_backward_vanishes_when_all_vocabulary_rows_are_equal():
    from oracle import lm_head as LH
    h, w, y = _lmh_case(seed=8)
    w_eq = np.tile(w[:1], (w.shape[0], 1))
    dh, _ = LH.edge_logprob_backward(h, w_eq, y, np.ones(len(y)))
    np.testing.assert_allclose(dh, 0.0, rtol=0, atol=1e-13)


def test_lm_head_rejects_labels_outside_the_vocabulary():
    from oracle import lm_head as LH
    h, w, y = _lmh_case()
    for bad in (w.shape[0], -1):
        y[0] = bad
        with pytest.raises(IndexError):
            LH.edge_logprob(h, w, y)


def test_lm_head_weight_grad_rows_equals_the_full_backward():
    from oracle import lm_head as LH
    h, w, y = _lmh_case(E=7, V=12, Hd=5, seed=9)
    g = np.random.default_rng(10).standard_normal(7)
    _, dw = LH.edge_logprob_backward(h, w, y, g)
    rows = np.array([y[0], 11, 0, y[3], 5])
    np.testing.assert_allclose(LH.weight_grad_rows(h, w, y, g, rows), dw[rows], rtol=0, atol=1e-13)


# ------------------------------------------------------------ bounded fragments

def test_fragments_single_fragment_when_the_cap_is_large():
    from oracle import fragments as OF
    t = W.tiny()
    frags = OF.plan_fragments(t.tree.seg_len, t.tree.parent, t.T)
    assert len(frags) == 1 and all(o for _, o in frags[0])
    assert OF.fragment_tokens(frags, t.tree.seg_len) == t.T


def test_fragments_hand_example():
    # root 64 -> children 32, 48 (-> grandchildren 16, 9), 17: the tiny tree, cap 130
    from oracle import fragments as OF
    lens = [64, 32, 48, 16, 9, 17]
    par = [-1, 0, 0, 2, 2, 0]
    frags = OF.plan_fragments(lens, par, 130)
    # 64+32 = 96; +48 > 130 -> new fragment {0, 2}, 112; +16 = 128; +9 > 130 -> new {0, 2, 4} = 121;
    # +17 > 130 -> new {0, 5} = 81
    assert frags == [[(0, True), (1, True)], [(0, False), (2, True), (3, True)],
                     [(0, False), (2, False), (4, True)], [(0, False), (5, True)]]
    assert OF.fragment_tokens(frags, lens) == 96 + 128 + 121 + 81
    OF.check_fragments(frags, lens, par, 130)


def test_fragments_are_valid_on_random_trees_and_workloads():
    from oracle import fragments as OF
    rng = np.random.default_rng(3)
    for _ in range(100):
        t = W.random_small_tree(rng, max_segments=12, max_len=30)
        longest_path = max(sum(int(t.seg_len[a]) for a in OT.ancestors(t.parent, s) + [s])
                           for s in range(t.num_segments))
        cap = int(rng.integers(longest_path, longest_path * 3 + 1))
        frags = OF.plan_fragments(t.seg_len, t.parent, cap)
        OF.check_fragments(frags, t.seg_len, t.parent, cap)
        assert OF.fragment_tokens(frags, t.seg_len) >= int(t.seg_len.sum())
    for name in ("agent", "long"):
        w = W.get(name)
        t = w.tree
        cap = 2 * max(sum(int(t.seg_len[a]) for a in OT.ancestors(t.parent, s) + [s]) for s in range(t.num_segments))
        frags = OF.plan_fragments(t.seg_len, t.parent, cap)
        OF.check_fragments(frags, t.seg_len, t.parent, cap)
        assert len(frags) > 1


def test_fragments_checker_catches_broken_covers():
    from oracle import fragments as OF
    lens, par = [64, 32, 48, 16, 9, 17], [-1, 0, 0, 2, 2, 0]
    good = OF.plan_fragments(lens, par, 130)
    bad_owner = [list(f) for f in good]
    bad_owner[1][0] = (0, True)  # the root owned twice
    bad_closure = [[(0, True), (1, True)], [(2, True), (3, True)], [(0, False), (2, False), (4, True)],
                   [(0, False), (5, True)]]
    for bad in (bad_owner, bad_closure):
        with pytest.raises(AssertionError):
            OF.check_fragments(bad, lens, par, 130)
    with pytest.raises(AssertionError):
        OF.check_fragments(good, lens, par, 120)


def test_fragments_accept_a_root_path_exactly_at_the_cap():
    from oracle import fragments as OF
    lens, par = [64, 32, 48, 16, 9, 17], [-1, 0, 0, 2, 2, 0]
    frags = OF.plan_fragments(lens, par, 128)  # 64 + 48 + 16: the longest root path
    OF.check_fragments(frags, lens, par, 128)
    assert [(3, True)] == [x for f in frags for x in f if x[0] == 3]


def test_fragments_reject_a_root_path_above_the_cap():
    from oracle import fragments as OF
    with pytest.raises(ValueError):
        OF.plan_fragments([64, 32, 48, 16, 9, 17], [-1, 0, 0, 2, 2, 0], 127)
