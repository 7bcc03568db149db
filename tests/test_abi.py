"""C-ABI checks that need no GPU: the library loads, exports every declared
symbol, builds plans bit-identical to the oracle's independent planner, and
rejects malformed input before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import workloads as W
from oracle import plan as OP

spc = pytest.importorskip("shared_prefix_causal_gb300")

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "shared_prefix_causal.h")


def test_library_exports_every_declared_symbol():
    decl = re.findall(r"SP_API\s+[\w\s\*]*?\b(sp_\w+)\s*\(", open(HEADER).read())
    assert len(decl) >= 9
    lib = ctypes.CDLL(spc.LIB_PATH)
    for name in decl:
        assert hasattr(lib, name), name
    assert set(decl) == set(spc.EXPORTED)


def _plan_tables(tree, tt, kb, order):
    p = spc.sp_tree_plan(tree.seg_start, tree.seg_len, tree.parent, tree.depth, tt, kb, order)
    return spc.sp_plan_view(p)


@pytest.mark.parametrize("name", ["tiny", "star", "forest", "agent", "long"])
@pytest.mark.parametrize("order", [0, 1])
def test_plan_bit_exact_on_configs(name, order):
    w = W.get(name)
    G = w.hq // w.hkv
    t = w.tree
    for tt in {128 // G, 16}:
        got = _plan_tables(t, tt, 128, order)
        want = OP.build(t.seg_start, t.seg_len, t.parent, tt, 128, order)
        for a, b in zip((got["tiles"], got["ranges"], got["bwd"]), want):
            assert a.dtype == np.int32
            assert np.array_equal(a, b)


@pytest.mark.parametrize("seed", range(100))
def test_plan_bit_exact_random(seed):
    rng = np.random.default_rng(seed)
    t = W.random_small_tree(rng, max_segments=12, max_len=40)
    tt, kb, order = int(rng.integers(1, 40)), int(rng.integers(1, 40)), int(rng.integers(0, 2))
    got = _plan_tables(t, tt, kb, order)
    want = OP.build(t.seg_start, t.seg_len, t.parent, tt, kb, order)
    for a, b in zip((got["tiles"], got["ranges"], got["bwd"]), want):
        assert np.array_equal(a, b)
    assert got["max_ranges_per_tile"] == int(want[0][:, 4].max())


def test_plan_matches_tiny_golden_file():
    from tests.test_oracle import _read_golden
    gold = _read_golden()
    t = W.tiny().tree
    got = _plan_tables(t, 32, 32, 0)
    tiles = [(int(s), int(a), int(b), [tuple(map(int, got["ranges"][r])) for r in range(rb, rb + rc)])
             for s, a, b, rb, rc in got["tiles"]]
    assert tiles == gold["tiles"]
    assert [tuple(map(int, b)) for b in got["bwd"]] == gold["bwd"]


def test_plan_order1_matches_tiny_golden_file():
    from tests.test_oracle import _read_golden
    got = _plan_tables(W.tiny().tree, 32, 32, 1)
    assert [tuple(map(int, r[:3])) for r in got["tiles"]] == _read_golden()["order1"]


def test_plan_matches_the_hand_worked_forest():
    from tests.test_oracle import FOREST_HAND as f
    p = spc.sp_tree_plan(f["seg_start"], f["seg_len"], f["parent"], f["depth"], 32, 32, 0)
    got = spc.sp_plan_view(p)
    tiles = [(int(s), int(a), int(b), [tuple(map(int, got["ranges"][r])) for r in range(rb, rb + rc)])
             for s, a, b, rb, rc in got["tiles"]]
    assert tiles == f["tiles"]
    assert [tuple(map(int, b)) for b in got["bwd"]] == f["bwd"]


def _desc(t):
    return [np.asarray(getattr(t, k)).copy() for k in ("seg_start", "seg_len", "parent", "depth")]


@pytest.mark.parametrize("mutate", [
    lambda a: a[1].__setitem__(2, 0),                       # empty segment
    lambda a: a[0].__setitem__(3, 100),                     # gap in packing
    lambda a: a[2].__setitem__(1, 3),                       # parent after child
    lambda a: a[2].__setitem__(0, 0),                       # first segment not a root
    lambda a: a[3].__setitem__(3, 1),                       # wrong depth
    lambda a: (a[2].__setitem__(5, 1), a[3].__setitem__(5, 2)),  # not preorder
    lambda a: a[2].__setitem__(4, -2),                      # parent below -1
    lambda a: a[0].__setitem__(3, 150),                     # a true gap (start after the previous end)
    lambda a: (a[1].__setitem__(4, 0), a[0].__setitem__(5, 160)),  # empty segment, packing consistent
])
def test_plan_rejects_invalid_tree(mutate):
    a = _desc(W.tiny().tree)
    mutate(a)
    with pytest.raises(spc.SPError) as e:
        spc.sp_tree_plan(*a, 32, 128, 0)
    assert e.value.code == -1


def _comb(levels):
    """A chain whose next node is each node's second child (after a one-token leaf): no root path
    merges, so the plan's interval tables grow with the square of the depth."""
    lens, pars, chain = [], [], -1
    for _ in range(levels):
        node = len(lens)
        lens.append(1)
        pars.append(chain)
        lens.append(1)
        pars.append(node)  # the leaf, first child of the node
        chain = node
    return W.tree_from_preorder(lens, pars)


def test_plan_refuses_trees_whose_tables_overflow_int32_indexing():
    t = _comb(33000)  # about 1.09e9 root-path intervals, over the 2^30 limit
    with pytest.raises(spc.SPError) as e:
        spc.sp_tree_plan(t.seg_start, t.seg_len, t.parent, t.depth, 128, 128, 0)
    assert e.value.code == -3
    small = _comb(300)
    got = _plan_tables(small, 128, 128, 0)
    want = OP.build(small.seg_start, small.seg_len, small.parent, 128, 128, 0)
    for a, b in zip((got["tiles"], got["ranges"], got["bwd"]), want):
        assert np.array_equal(a, b)
    assert got["max_ranges_per_tile"] == 300
    # the fragment planner refuses the same deep comb for the same reason, and plans the small one
    with pytest.raises(RuntimeError, match="status -3"):
        spc.fragment_plan(t, 10 ** 9)
    frag = spc.fragment_plan(small, 10 ** 6)
    assert frag["num_fragments"] == 1 and frag["fragment_tokens"] == small.total_tokens


def test_upload_refuses_plans_whose_forward_block_lists_could_overflow():
    """One 600K-token sequence cut into 1-token tiles: its tiles' ranges hold about 1.4e9 blocks of
    128 keys.  The plan itself is fine; its upload is refused before any CUDA call."""
    T = 600_000
    p = spc.sp_tree_plan([0], [T], [-1], [0], 1, 128, 0)
    assert spc.sp_plan_device_bytes(p) == 0
    assert spc._c_plan_upload(p.handle, None) == -3  # refused before any CUDA call
    t = W.tiny().tree
    assert spc.sp_plan_device_bytes(spc.sp_tree_plan(t.seg_start, t.seg_len, t.parent, t.depth, 128, 128, 0)) > 0


def test_merged_backward_blocks_through_the_binding():
    """sp_plan_bwd_blocks on the CPU (no upload needed): the tiny tree's six canonical key blocks
    become three, every key once, each block's run that of its first key; null pointers refused."""
    t = W.tiny().tree
    p = spc.sp_tree_plan(t.seg_start, t.seg_len, t.parent, t.depth, 32, 128, 0)
    m, v = spc.sp_plan_bwd_blocks(p), spc.sp_plan_view(p)
    rows, key_end = m["rows"], m["key_end"]
    assert len(v["bwd"]) == 6 and len(rows) == 3
    seen = np.zeros(t.total_tokens, dtype=np.int64)
    for seg, k0, k1, q0, q1 in rows.tolist():
        assert q0 == k0 and q1 == key_end[k0] and (key_end[k0:k1] <= q1).all()
        seen[k0:k1] += 1
    assert (seen == 1).all()
    for seg, k0, k1, q0, q1 in v["bwd"].tolist():
        assert (key_end[k0:k1] == q1).all()
    out = ctypes.POINTER(ctypes.c_int32)()
    n = ctypes.c_int32()
    assert spc._c_plan_bwd_blocks(p.handle, None, ctypes.byref(n), ctypes.byref(out)) == -2
    assert spc._c_plan_bwd_blocks(None, ctypes.byref(out), ctypes.byref(n), ctypes.byref(out)) == -2


def test_plan_rejects_bad_arguments():
    a = _desc(W.tiny().tree)
    for tt, kb, order in ((0, 128, 0), (32, 0, 0), (32, 128, 2)):
        with pytest.raises(spc.SPError) as e:
            spc.sp_tree_plan(*a, tt, kb, order)
        assert e.value.code == -2


def test_empty_tree_gives_empty_plan():
    e = np.zeros(0, dtype=np.int32)
    info = spc.sp_plan_view(spc.sp_tree_plan(e, e, e, e, 32, 128, 0))
    assert info["tiles"].shape == (0, 5) and info["bwd"].shape == (0, 5)


def test_status_strings_and_workspace_size():
    assert spc.sp_status_string(0) == "ok"
    assert "preorder" in spc.sp_status_string(-1)
    assert spc.sp_status_string(12345) == "unknown status"
    assert spc.sp_tree_attn_bwd_workspace_bytes(spc.SP_F32, 0, 4, 64) == 0
    n = spc.sp_tree_attn_bwd_workspace_bytes(spc.SP_BF16, 1000, 8, 128)
    assert n >= 1000 * 8 * 4 and n % 256 == 0


def test_attention_argument_checks_fail_before_device_work():
    """Bad arguments come back as status codes; no pointer is dereferenced."""
    t = W.tiny().tree
    p = spc.sp_tree_plan(t.seg_start, t.seg_len, t.parent, t.depth, 64, 128, 0)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the checks fail first
    f = spc._c_fwd
    args = lambda dtype, T, Hq, Hkv, D, ptr=fake: (p.handle, dtype, ptr, ptr, ptr, ptr, ptr, T, Hq, Hkv, D,  # noqa
                                                   0.125, None, None)
    assert f(*args(0, 186, 2, 2, 96)) == -3          # head_dim
    assert f(*args(0, 186, 6, 4, 64)) == -3          # Hq % Hkv
    assert f(*args(0, 186, 32, 2, 64)) == -3         # G = 16
    assert f(*args(7, 186, 2, 2, 64)) == -3          # dtype
    assert f(*args(0, 185, 2, 2, 64)) == -2          # T mismatch
    assert f(*args(0, 186, 2, 2, 64, ctypes.c_void_p((1 << 20) + 8))) == -4  # alignment
    assert f(*args(0, 186, 2, 2, 64)) == -9          # plan not uploaded
    assert f(None, 0, fake, fake, fake, fake, fake, 186, 2, 2, 64, 0.125, None, None) == -2
    b = spc._c_bwd
    assert b(p.handle, 0, fake, fake, fake, fake, fake, fake, fake, fake, fake, None, 0, 186, 2, 2, 64, 0.125,
             None, None) == -8
    assert b(p.handle, 0, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 1 << 30, 186, 2, 2, 64,
             0.125, None, None) == -9
    g = spc._c_gather
    assert g(0, fake, 186, 256, fake, 0, fake, None, None) == 0       # E == 0: no-op
    assert g(0, fake, 186, 3, fake, 4, fake, None, None) == -3        # row not a multiple of 16 bytes
    assert g(0, fake, 186, 256, fake, -1, fake, None, None) == -2
    assert g(0, ctypes.c_void_p((1 << 20) + 2), 186, 256, fake, 4, fake, None, None) == -4


def test_zero_sized_calls_are_no_ops_before_any_device_work():
    """An empty tree (T = 0), no actions (E = 0) or no requested outputs return SP_OK at once:
    nothing is read, written or launched, so null pointers are fine and no GPU is needed."""
    e = np.zeros(0, dtype=np.int32)
    p = spc.sp_tree_plan(e, e, e, e, 32, 128, 0)  # never uploaded
    n9 = [None] * 9
    for dtype in (spc.SP_BF16, spc.SP_F32):
        assert spc._c_fwd(p.handle, dtype, *n9[:5], 0, 32, 8, 128, 0.1, None, None) == 0
        for fn in (spc._c_bwd, spc._c_bwd_det):
            assert fn(p.handle, dtype, *n9, None, 0, 0, 32, 8, 128, 0.1, None, None) == 0
        assert spc._c_bwd_noalloc(p.handle, dtype, *n9, 0, 32, 8, 128, 0.1, None, None) == 0
        assert spc._c_gather_bwd(dtype, None, 0, 256, None, 0, None, None, 0, None, None) == 0
    assert spc._c_lmh(spc.SP_BF16, None, 0, 64, None, 96, None, None, None, None, 0, None, None) == 0
    # backward with neither gradient requested
    assert spc._c_lmh_bwd(spc.SP_BF16, None, 5, 64, None, 96, None, None, None, None, None, None, 0, None,
                          None) == 0
    # a non-empty plan still refuses T = 0
    t = W.tiny().tree
    q = spc.sp_tree_plan(t.seg_start, t.seg_len, t.parent, t.depth, 64, 128, 0)
    assert spc._c_fwd(q.handle, spc.SP_BF16, *n9[:5], 0, 2, 2, 64, 0.1, None, None) == -2


def test_bench_traffic_is_null_when_kernel_sources_change(monkeypatch):
    import bench
    assert bench.measured_traffic("nowhere", "bwd_tc_kernel", 1)[0] is None  # never captured
    for cfg, ks in bench.MEASURED_TRAFFIC.items():
        assert ks["units"] > 0
        for k, (nbytes, digest) in ((k, v) for k, v in ks.items() if k != "units"):
            assert len(digest) == 16 and nbytes > 0
    # every bench workload has a capture of its own or of a reduced twin
    for cfg in W.CONFIGS:
        assert cfg in bench.MEASURED_TRAFFIC or bench.TRAFFIC_SCALED_FROM[cfg] in bench.MEASURED_TRAFFIC
    monkeypatch.setitem(bench.MEASURED_TRAFFIC, "agent_small",
                        {"units": 10, "bwd_tc_kernel": (1.0, "0" * 16)})
    assert bench.measured_traffic("agent_small", "bwd_tc_kernel", 10)[0] is None
    assert bench.measured_traffic("agent", "bwd_tc_kernel", 30)[0] is None
    monkeypatch.setitem(bench.MEASURED_TRAFFIC, "agent_small",
                        {"units": 10, "bwd_tc_kernel": (7.0, bench.sources_digest("bwd_tc_kernel"))})
    assert bench.measured_traffic("agent_small", "bwd_tc_kernel", 10)[0] == 7
    nbytes, how = bench.measured_traffic("agent", "bwd_tc_kernel", 30)
    assert nbytes == 21 and "agent_small" in how and "x3.000" in how


# ------------------------------------------------------------ bounded fragments

def _oracle_frag_tables(tree, cap):
    from oracle import fragments as OF
    frags = OF.plan_fragments(tree.seg_len, tree.parent, cap)
    seg = [a for f in frags for a, _ in f]
    owned = [int(o) for f in frags for _, o in f]
    offsets = np.cumsum([0] + [len(f) for f in frags])
    return frags, np.array(seg), np.array(owned), offsets


def _longest_path(tree):
    from oracle import tree as OT
    return max(sum(int(tree.seg_len[a]) for a in OT.ancestors(tree.parent, s) + [s])
               for s in range(tree.num_segments))


@pytest.mark.parametrize("name", ["tiny", "star", "forest", "agent", "long"])
def test_fragment_plan_bit_exact_vs_oracle(name):
    w = W.get(name)
    lp = _longest_path(w.tree)
    for cap in (lp, 2 * lp, w.T):
        got = spc.fragment_plan(w.tree, cap)
        frags, seg, owned, offsets = _oracle_frag_tables(w.tree, cap)
        assert got["num_fragments"] == len(frags)
        assert np.array_equal(got["offsets"], offsets)
        assert np.array_equal(got["seg"], seg) and np.array_equal(got["owned"], owned)
        assert got["fragment_tokens"] == sum(int(w.tree.seg_len[a]) for a in seg)
        assert got["physical_tokens"] == w.T


def test_fragment_plan_random_trees_and_fragment_trees_are_valid():
    rng = np.random.default_rng(21)
    for _ in range(150):
        t = W.random_small_tree(rng, max_segments=14, max_len=40)
        lp = _longest_path(t)
        cap = int(rng.integers(lp, 3 * lp + 1))
        got = spc.fragment_plan(t, cap)
        _, seg, owned, offsets = _oracle_frag_tables(t, cap)
        assert np.array_equal(got["seg"], seg) and np.array_equal(got["owned"], owned)
        assert np.array_equal(got["offsets"], offsets)
        for f in range(got["num_fragments"]):
            start, ln, par, dep, segs, own = spc.fragment_tree(got, f, t)
            assert int(ln.sum()) == int(got["tokens"][f]) <= cap
            # a valid packed tree of its own: the planner accepts it
            spc.sp_tree_plan(start, ln, par, dep, 4, 16, 0)


def test_fragment_plan_rejections():
    w = W.get("tiny")
    with pytest.raises(RuntimeError, match="fragment token cap"):
        spc.fragment_plan(w.tree, _longest_path(w.tree) - 1)
    with pytest.raises(RuntimeError):
        spc.fragment_plan(w.tree, 0)
    bad_parent = np.array(w.tree.parent).copy()
    bad_parent[3] = 4  # parent after the child: not a preorder
    with pytest.raises(RuntimeError):
        spc.sp_fragment_plan(w.tree.seg_start, w.tree.seg_len, bad_parent, w.tree.depth, 1000)
    empty = spc.sp_fragment_plan([], [], [], [], 10)
    assert empty["num_fragments"] == 0 and empty["fragment_tokens"] == 0


def test_vocab_head_gather_bwd_and_deterministic_argument_checks():
    """Status codes for the newer entry points; every case fails (or returns) before device work."""
    fake = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 8)
    lp = spc._c_lmh
    ws = spc.sp_edge_logprob_workspace_bytes(300, 1000)
    assert ws >= 8 * 300 * 4 + 4 * 300
    ok = lambda **kw: dict(dict(dtype=0, h=fake, E=300, Hd=128, w=fake, V=1000, y=fake, lp=fake, lse=fake,  # noqa
                                ws=fake, wsb=ws), **kw)
    call = lambda a: lp(a["dtype"], a["h"], a["E"], a["Hd"], a["w"], a["V"], a["y"], a["lp"], a["lse"],  # noqa
                        a["ws"], a["wsb"], None, None)
    assert call(ok(dtype=7)) == -2
    assert call(ok(dtype=1)) == -3                    # fp32 inputs: not supported here
    assert call(ok(E=-1)) == -2 and call(ok(V=0)) == -2 and call(ok(Hd=0)) == -2
    assert call(ok(Hd=12)) == -3                      # rows not a multiple of 16 bytes
    assert call(ok(E=0)) == 0                         # no actions: nothing to do
    assert call(ok(y=None)) == -2
    assert call(ok(h=mis)) == -4
    assert call(ok(wsb=ws - 1)) == -8
    assert call(ok(ws=ctypes.c_void_p((1 << 20) + 16))) == -4  # workspace not 256-byte aligned
    lb = spc._c_lmh_bwd
    wsb = spc.sp_edge_logprob_bwd_workspace_bytes(300, 1000)
    assert wsb >= 2 * 300 * 1000
    bcall = lambda E=300, Hd=128, V=1000, dh=fake, dw=fake, b=wsb, h=fake: lb(  # noqa
        0, h, E, Hd, fake, V, fake, fake, fake, dh, dw, fake, b, None, None)
    assert bcall(V=1004) == -3                        # V % 8
    assert bcall(dh=None, dw=None) == 0               # nothing requested
    assert bcall(E=0, dw=None) == 0                   # no actions, no weight gradient requested
    assert bcall(b=wsb - 1) == -8
    assert bcall(h=mis) == -4
    assert spc.sp_edge_logprob_bwd_workspace_bytes(-1, 8) == 0
    gb = spc._c_gather_bwd
    gws = spc.sp_edge_gather_bwd_workspace_bytes(186, 8)
    assert gb(0, fake, 8, 256, fake, 0, fake, fake, gws, None, None) == 0       # T == 0
    assert gb(0, fake, 8, 12, fake, 186, fake, fake, gws, None, None) == -3     # hidden_dim % 8
    assert gb(0, fake, -1, 256, fake, 186, fake, fake, gws, None, None) == -2
    assert gb(0, fake, 8, 256, fake, 186, fake, fake, gws - 1, None, None) == -8
    assert gb(0, fake, 8, 256, fake, 186, mis, fake, gws, None, None) == -4
    assert gb(5, fake, 8, 256, fake, 186, fake, fake, gws, None, None) == -3
    t = W.tiny().tree
    p = spc.sp_tree_plan(t.seg_start, t.seg_len, t.parent, t.depth, 64, 128, 0)
    d = spc._c_bwd_det
    assert d(p.handle, 0, fake, fake, fake, fake, fake, fake, fake, fake, fake, None, 0, 186, 2, 2, 64, 0.125,
             None, None) == -8
    assert d(p.handle, 0, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 1 << 30, 186, 2, 2, 64,
             0.125, None, None) == -9
    assert d(p.handle, 0, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 1 << 30, 186, 2, 2, 96,
             0.125, None, None) == -3
    assert "cap" in spc.sp_status_string(spc.SP_ERR_CAP)


def test_fragment_tokens_index_the_whole_tree():
    w = W.get("star")
    frag = spc.fragment_plan(w.tree, 3034)
    owned_total = np.zeros(w.T, dtype=np.int64)
    for f in range(frag["num_fragments"]):
        idx, own = spc.fragment_tokens(frag, f, w.tree)
        assert len(idx) == int(frag["tokens"][f]) and len(set(idx.tolist())) == len(idx)
        start, ln, par, dep, segs, _ = spc.fragment_tree(frag, f, w.tree)
        # the fragment's packed layout maps segment by segment onto the tree's tokens
        for s_, st_ in zip(segs, start):
            assert idx[st_] == int(w.tree.seg_start[s_])
        np.add.at(owned_total, idx[own], 1)
    assert (owned_total == 1).all()  # every token owned exactly once


def test_plan_upload_to_checks():
    t = W.tiny().tree
    p = spc.sp_tree_plan(t.seg_start, t.seg_len, t.parent, t.depth, 64, 128, 0)
    n = spc.sp_plan_device_bytes(p)
    assert n > 0 and n % 256 == 0
    assert spc._c_plan_bytes(None) == 0
    fake = ctypes.c_void_p(1 << 20)
    assert spc._c_plan_upload_to(p.handle, None, n, None) == -2
    assert spc._c_plan_upload_to(None, fake, n, None) == -2
    assert spc._c_plan_upload_to(p.handle, ctypes.c_void_p((1 << 20) + 16), n, None) == -4
    assert spc._c_plan_upload_to(p.handle, fake, n - 1, None) == -8


# ------------------------------------------------------------ bench host helpers

def _golden_value(key):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_plan.txt")
    for line in open(path):
        parts = line.split()
        if len(parts) >= 2 and parts[0] == key:
            return int(parts[1])
    raise KeyError(key)


def test_bench_useful_pairs_matches_the_hand_derived_count():
    import bench
    assert bench.useful_pairs(W.get("tiny").tree) == _golden_value("pairs")


def test_bench_tile_efficiency_by_hand_on_a_single_segment():
    """One 300-token segment, G = 4 (32-token tiles, 16-token backward blocks): computed pairs by hand."""
    import bench
    t = W.tree_from_preorder([300], [-1])
    p = spc.sp_tree_plan(t.seg_start, t.seg_len, t.parent, t.depth, 32, 128, 0)
    pairs = 300 * 301 // 2
    # forward: tile k covers tokens [32k, min(32k+32, 300)) and reads keys [0, q_end) in 128-key blocks
    fwd = sum(((min(32 * k + 32, 300) + 127) // 128) * 128 * 32 for k in range(10))
    # backward: key block [128b, ...) walks queries [128b, 300) in 16-token blocks of 128 keys
    bwd = sum(((300 - 128 * b + 15) // 16) * 16 * 128 for b in range(3))
    eff = bench.tile_efficiency(spc, p, 4, pairs)
    assert eff == {"fwd": round(pairs / fwd, 4), "bwd": round(pairs / bwd, 4)}


def test_bench_fragment_summary():
    import bench
    out = bench.fragment_summary(spc, W.get("tiny"), 130)
    assert out["fragments"] == 4 and out["fragment_tokens"] == 426 and out["physical_tokens"] == 186
    assert out["duplication"] == round(426 / 186, 4)
    # a cap below the longest root path (64 + 48 + 16 = 128 tokens) is doubled until it holds it
    out = bench.fragment_summary(spc, W.get("tiny"), 10)
    assert out["cap"] == 160 and out["cap_asked"] == 10 and out["longest_root_path"] == 128
    assert out == {**bench.fragment_summary(spc, W.get("tiny"), 160), "cap_asked": 10, "longest_root_path": 128,
                   "plan_ms": out["plan_ms"]}


def test_bench_clock_sampler_keeps_only_the_timed_window(tmp_path):
    """nvidia-smi lines (timestamp first) outside the timed region are dropped; throttle reasons are
    collected from the kept lines only; the median SM clock is over the kept lines."""
    import datetime
    import bench

    def line(t, sm, reasons=("Not Active",) * 4):
        ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return ", ".join([ts, "0", str(sm), "2070", "900.00", "0x0000000000000000", *reasons]) + "\n"

    t0 = 1_800_000_000.0
    csv = tmp_path / "clocks.csv"
    csv.write_text(line(t0 - 2.0, 800, ("Active", "Not Active", "Not Active", "Not Active"))  # before
                   + line(t0 + 0.1, 2070) + line(t0 + 0.2, 2055)
                   + line(t0 + 0.3, 2040, ("Not Active", "Not Active", "Not Active", "Active"))
                   + "garbage line\n"
                   + line(t0 + 5.0, 1000, ("Not Active", "Active", "Not Active", "Not Active")))  # after

    class FakeProc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    cs = bench.ClockSampler(0)
    cs.proc, cs.path = FakeProc(), str(csv)
    cs.mark(t0, t0 + 0.4)
    got = cs.stop()
    assert got == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert not csv.exists()


def test_bench_clock_sampler_without_nvidia_smi_reports_nothing():
    import bench
    assert bench.ClockSampler(0).stop() is None


@pytest.mark.parametrize("content,want", [
    ({"hbm_gbs": 7000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1750.0},
     {"burst": (2000.0, "measured"), "sustained": (1750.0, "measured"), "hbm": (7000.0, "measured")}),
    ({"gb300": {"hbm_gbs": {"value": 7100}, "bf16_tflops": {"median": 1980.5}}, "clocks": {"sm_mhz": 2070}},
     {"burst": (1980.5, "measured"), "sustained": (1700.0, "fallback"), "hbm": (7100.0, "measured")}),
    ({"bf16_tflops": None, "hbm_gbs": "n/a"},
     {"burst": (1900.0, "fallback"), "sustained": (1700.0, "fallback"), "hbm": (6800.0, "fallback")}),
    ("not json", {"burst": (1900.0, "fallback"), "sustained": (1700.0, "fallback"), "hbm": (6800.0, "fallback")}),
    (None, {"burst": (1900.0, "fallback"), "sustained": (1700.0, "fallback"), "hbm": (6800.0, "fallback")}),
])
def test_bench_peaks_from_the_measured_file_else_the_fallback(tmp_path, content, want):
    import json
    import bench
    path = tmp_path / "peaks.json"
    if content is not None:
        path.write_text(content if isinstance(content, str) else json.dumps(content))
    assert bench.resolve_peaks(*bench.load_peaks(str(path))) == want


def test_bench_cta_tail_stats_by_hand():
    """Two SMs, two CTAs each: SM 0 busy [0, 100) and [100, 150), SM 1 busy [0, 80) and [80, 120); the
    launch spans 150; SM 1 idles 30 after its last CTA: tail idle 30 / (150 x 2), busy 270 / 300."""
    import bench
    rec = np.array([[0, 100, 0, 0], [0, 80, 1, 0], [100, 150, 0, 0], [80, 120, 1, 0], [0, 0, 0, 0]],
                   dtype=np.int64)  # the last row: a CTA past the buffer records nothing
    out = bench.cta_tail_stats(rec)
    assert out["ctas"] == 4 and out["sms"] == 2
    assert out["tail_idle_frac"] == pytest.approx(0.1) and out["busy_frac"] == pytest.approx(0.9)
    assert out["longest_cta_us"] == pytest.approx(0.1) and out["last_sm_idle_us"] == pytest.approx(0.03)
