"""The planner tests catch planted mistakes in the library's host C++.

Each case plants one plausible mistake in a copy of ``plan.cpp`` (tree
validation, tiling, range merging, ordering, the backward table) or
``fragments.cpp`` (the bounded fragment planner).  The copy is built with g++
into a small host-only library, together with ``tests/c/planner_shim.cpp``.
The case then runs the checks the planner's parity tests make (hand-derived
plans, the oracle's planner and fragment planner on random trees, accepted and
refused trees) and expects at least one to fail.  No GPU, no CUDA.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import workloads as W
from oracle import fragments as OF
from oracle import plan as OP
from oracle import tree as OT

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "shared_prefix_causal_gb300", "csrc")
SHIM = os.path.join(ROOT, "tests", "c", "planner_shim.cpp")

pytestmark = pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")

# (file, text in it, replacement, what the mistake is)
MUTANTS = [
    ("plan.cpp", "if (!v.empty() && v.back().second == x.first)", "if (false)", "touching ranges not merged"),
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


class _Desc(ctypes.Structure):
    _fields_ = [("num_segments", ctypes.c_int32), ("total_tokens", ctypes.c_int32)] + \
               [(n, ctypes.POINTER(ctypes.c_int32)) for n in ("seg_start", "seg_len", "parent", "depth")]


class _FragInfo(ctypes.Structure):
    _fields_ = [("num_fragments", ctypes.c_int32), ("num_entries", ctypes.c_int32),
                ("physical_tokens", ctypes.c_int64), ("fragment_tokens", ctypes.c_int64)] + \
               [(n, ctypes.POINTER(ctypes.c_int32)) for n in ("offsets", "tokens", "seg", "owned", "local_parent",
                                                              "local_start")]


class Host:
    """ctypes view of one host-only build."""

    def __init__(self, path):
        self.lib = ctypes.CDLL(path)
        self.lib.shim_plan.restype = ctypes.c_void_p
        self.lib.shim_plan.argtypes = [ctypes.POINTER(_Desc), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.POINTER(ctypes.c_int32)]
        self.lib.shim_rows.restype = ctypes.c_int32
        self.lib.shim_rows.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.POINTER(ctypes.c_int32))]
        self.lib.shim_free.argtypes = [ctypes.c_void_p]
        self.lib.sp_fragment_plan.argtypes = [ctypes.POINTER(_Desc), ctypes.c_int64, ctypes.POINTER(ctypes.c_void_p)]
        self.lib.sp_fragment_view.argtypes = [ctypes.c_void_p, ctypes.POINTER(_FragInfo)]
        self.lib.sp_fragment_destroy.argtypes = [ctypes.c_void_p]

    @staticmethod
    def _desc(st, ln, par, dep, total=None):
        arrs = [np.ascontiguousarray(np.asarray(a, dtype=np.int32)) for a in (st, ln, par, dep)]
        total = int(arrs[1].sum()) if total is None else total
        return _Desc(len(arrs[0]), total, *[a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) for a in arrs]), arrs

    def plan(self, st, ln, par, dep, tile, kvb, order, total=None):
        d, keep = self._desc(st, ln, par, dep, total)
        rc = ctypes.c_int32()
        h = self.lib.shim_plan(ctypes.byref(d), tile, kvb, order, ctypes.byref(rc))
        if rc.value:
            return rc.value
        out = []
        for which, w in ((0, 5), (1, 2), (2, 5)):
            ptr = ctypes.POINTER(ctypes.c_int32)()
            n = self.lib.shim_rows(h, which, ctypes.byref(ptr))
            out.append(np.ctypeslib.as_array(ptr, shape=(n * w,)).reshape(n, w).copy() if n else
                       np.zeros((0, w), dtype=np.int32))
        self.lib.shim_free(h)
        return tuple(out)

    def fragments(self, st, ln, par, dep, cap):
        d, keep = self._desc(st, ln, par, dep)
        h = ctypes.c_void_p()
        rc = self.lib.sp_fragment_plan(ctypes.byref(d), cap, ctypes.byref(h))
        if rc:
            return rc
        info = _FragInfo()
        assert self.lib.sp_fragment_view(h, ctypes.byref(info)) == 0
        get = lambda p, n: np.ctypeslib.as_array(p, shape=(n,)).copy() if n else np.zeros(0, np.int32)  # noqa: E731
        ne, nf = info.num_entries, info.num_fragments
        out = {k: get(getattr(info, k), ne) for k in ("seg", "owned", "local_parent", "local_start")}
        out["offsets"], out["tokens"] = get(info.offsets, nf + 1), get(info.tokens, nf)
        self.lib.sp_fragment_destroy(h)
        return out


_CXX = ["g++", "-std=c++17", "-O0", "-fPIC", "-fvisibility=hidden", "-I", CSRC]


def _compile(src, obj):
    subprocess.run(_CXX + ["-c", str(src), "-o", str(obj)], check=True, capture_output=True, text=True)
    return str(obj)


def _build(objs, d, mutant=None):
    """A host-only library: the original objects, with the mutated file (if any) recompiled."""
    d.mkdir()
    parts = dict(objs)
    if mutant:
        f, old, new = mutant[:3]
        text = open(os.path.join(CSRC, f), encoding="utf-8").read()
        assert text.count(old) == 1, f"{f}: the planted text must occur exactly once: {old!r}"
        (d / f).write_text(text.replace(old, new))
        parts[f] = _compile(d / f, d / (f + ".o"))
    out = str(d / "libhost.so")
    subprocess.run(["g++", "-shared", *parts.values(), "-o", out], check=True, capture_output=True, text=True)
    return Host(out)


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
    objs = {f: _compile(os.path.join(CSRC, f), d / (f + ".o")) for f in ("plan.cpp", "fragments.cpp")}
    objs["shim"] = _compile(SHIM, d / "shim.o")
    return d, objs


def test_unmutated_host_code_passes_the_battery(objects):
    d, objs = objects
    _battery(_build(objs, d / "original"))


@pytest.mark.parametrize("mutant", MUTANTS, ids=[f"{m[0]}: {m[3]}" for m in MUTANTS])
def test_planted_host_mistake_is_caught(objects, mutant):
    d, objs = objects
    host = _build(objs, d / f"m{MUTANTS.index(mutant)}", mutant)
    with pytest.raises(AssertionError):
        _battery(host)
