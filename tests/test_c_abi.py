"""The C ABI used from plain C, with no Python in between.

``tests/c/abi_from_c.c`` is compiled as strict C99 against
``include/shared_prefix_causal.h`` and linked with the library.  It plans
trees fed on its stdin and prints the tables.  They must equal the oracle's
planner and fragment planner.  The header must also compile as C++.  No GPU
call is made.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import workloads as W
from oracle import fragments as OF
from oracle import plan as OP
from oracle import tree as OT

spc = pytest.importorskip("shared_prefix_causal_gb300")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
SOURCE = os.path.join(ROOT, "tests", "c", "abi_from_c.c")

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    libdir = os.path.dirname(spc.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("c_abi") / "abi_from_c")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, SOURCE,
                    "-L", libdir, "-l:" + os.path.basename(spc.LIB_PATH), "-Wl,-rpath," + libdir, "-o", exe],
                   check=True, capture_output=True, text=True)
    return exe


def _run(exe, tree, tile, kvb, order, cap):
    n = len(tree.seg_len)
    lines = [str(n)] + [f"{int(tree.seg_start[s])} {int(tree.seg_len[s])} {int(tree.parent[s])} {int(tree.depth[s])}"
                        for s in range(n)] + [f"{tile} {kvb} {order} {cap}"]
    out = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True).stdout
    got = {"T": [], "R": [], "B": [], "O": [], "F": [], "M": [], "E": []}
    for line in out.splitlines():
        tag, *vals = line.split()
        if tag in ("plan", "frag", "E"):
            got[tag] = [int(x) for x in vals]
        else:
            got[tag].append([int(x) for x in vals])
    return got


def _longest_path(t):
    return max(sum(int(t.seg_len[a]) for a in OT.ancestors(t.parent, s) + [s]) for s in range(t.num_segments))


def _check(got, t, tile, kvb, order, cap):
    tiles, ranges, bwd = OP.build(t.seg_start, t.seg_len, t.parent, tile, kvb, order)
    assert got["plan"][0] == 0
    assert np.array_equal(np.array(got["T"], dtype=np.int32).reshape(-1, 5), tiles)
    assert np.array_equal(np.array(got["R"], dtype=np.int32).reshape(-1, 2), ranges)
    assert np.array_equal(np.array(got["B"], dtype=np.int32).reshape(-1, 5), bwd)
    # the merged backward key blocks read through sp_plan_bwd_blocks, held to their reading
    # against the oracle's canonical table
    from test_device_tables import check_merged_blocks
    rows = np.array(got["M"], dtype=np.int64).reshape(-1, 5)
    runs = rows[:, 4] - rows[:, 3]
    check_merged_blocks(int(t.seg_len.sum()), {"bwd": bwd, "bwd_merged": rows, "key_end": np.array(got["E"]),
                                               "runm_sum": int(runs.sum()),
                                               "runm_max": int(runs.max()) if len(runs) else 0}, block=kvb)
    frags = OF.plan_fragments(t.seg_len, t.parent, cap)
    assert got["frag"][:3] == [0, len(frags), sum(len(f) for f in frags)]
    assert got["frag"][3:] == [int(t.seg_len.sum()), OF.fragment_tokens(frags, t.seg_len)]
    assert [o for (o,) in got["O"]] == list(np.cumsum([0] + [len(f) for f in frags]))
    assert [(s, o) for s, o, _, _ in got["F"]] == [(a, int(own)) for f in frags for a, own in f]


def test_header_compiles_as_cpp():
    if shutil.which("g++") is None:
        pytest.skip("needs g++")
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only", "-x", "c++",
                    os.path.join(INCLUDE, "shared_prefix_causal.h")], check=True, capture_output=True, text=True)


def test_tiny_tree_from_c_matches_the_oracle_and_the_golden_plan(driver):
    t = W.tiny().tree
    got = _run(driver, t, 32, 32, 0, 130)
    _check(got, t, 32, 32, 0, 130)
    assert got["plan"][1:] == [8, 14, 8, 3]


def test_random_trees_from_c_match_the_oracle(driver):
    rng = np.random.default_rng(41)
    for _ in range(30):
        t = W.random_small_tree(rng, max_segments=12, max_len=40)
        tile, kvb, order = int(rng.integers(1, 40)), int(rng.integers(1, 40)), int(rng.integers(0, 2))
        lp = _longest_path(t)
        cap = int(rng.integers(lp, 3 * lp + 1))
        _check(_run(driver, t, tile, kvb, order, cap), t, tile, kvb, order, cap)


def test_agent_tree_from_c_matches_the_oracle(driver):
    t = W.get("agent").tree
    cap = 2 * _longest_path(t)
    _check(_run(driver, t, 32, 128, 0, cap), t, 32, 128, 0, cap)


def test_invalid_tree_from_c_is_refused(driver):
    t = W.tiny().tree
    bad = W.tiny().tree
    bad.parent = np.array(t.parent).copy()
    bad.parent[3] = 4  # parent after child
    got = _run(driver, bad, 32, 32, 0, 130)
    assert got["plan"][0] == -1 and got["T"] == [] and got["frag"][0] != 0
