"""The tables the kernels read, checked on the CPU.

At upload the library builds, from the canonical plan, the forward's work
list and the backward's launch order:
  * pairs [n][4] = {tile_a, tile_b or -1, first entry, entry count}: tiles
    2i and 2i+1 of the schedule share one CTA;
  * pblk [m][8] = {kb, nb, end_a or 0, end_b or 0, 0, 0, causal bits, 0}: the
    pair's 128-key blocks merged by start, as runs of nb blocks kb, kb + 128,
    ...  Tile t reads keys [kb, min(kb + 128, end_t)) of a block whose end_t is
    non-zero, and only keys j <= its query i when bit t is set;
  * bwd_sched: the backward table's rows in launch order (latest run end
    first, longest run first within a run end), with the runs' sum and maximum.
  * bwd_merged, key_end: the tensor-core backward's key blocks, in the same
    launch order.  Every key is in exactly one block; a block walks the query
    run [first key, run end of its first key) and each of its keys is masked
    with its own run end key_end (the subtree end of its segment), never past
    the block's.  A block of fewer than 128 keys ends where the next key
    belongs to no segment of its first key's subtree.
  * quads [n][6] = {a0, a1, b0, b1 (or -1), first entry, entry count}: the
    paired-SM forward's work items.  A couple (a0, a1) or (b0, b1) is two
    consecutive tiles of one segment (offsets 2i and 2i + 1; a segment's last
    odd tile alone), couples in the order of their first tiles in the
    schedule, two per quad;
  * qblk [m][8] = {kb, nb, end a0, a1, b0, b1 (or 0), causal bits, 0}: the
    quad's block runs, read as the pairs' runs are.
These checks hold the tables to that reading, to the forward kernels' own
validity tests, and to the canonical plan.  The tables come from the host-only
build of the planner (no CUDA).
"""
import shutil

import numpy as np
import pytest

import workloads as W

from host_planner import Host, build_host_library, original_objects

pytestmark = pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
BLOCK = 128


def _merge(ivs):
    out = []
    for a, b in sorted(ivs):
        if out and out[-1][1] == a:
            out[-1] = (out[-1][0], b)
        else:
            out.append((a, b))
    return out


def expand_runs(runs):
    """Runs [r][8] = {kb, nb, end[4], causal bits, 0} as one row per 128-key block: {kb, end[4], bits}."""
    rows = []
    for kb, nb, e0, e1, e2, e3, bits, zero in runs.tolist():
        assert zero == 0 and nb >= 1
        rows += [[kb + BLOCK * i, e0, e1, e2, e3, bits] for i in range(nb)]
    return np.array(rows, dtype=np.int64).reshape(-1, 6)


def check_runs_as_the_kernels_do(T, runs, present):
    """The forward kernels' own test of a work item's runs (check_runs in pipeline.cuh)."""
    kb, nb = runs[:, 0].astype(np.int64), runs[:, 1].astype(np.int64)
    last = kb + BLOCK * (nb - 1)
    assert ((nb >= 1) & (kb >= 0) & (last < T)).all()
    for s_ in range(4):
        end = runs[:, 2 + s_].astype(np.int64)
        bit = (runs[:, 6] >> s_) & 1
        assert not bit[end == 0].any()
        if not present[s_]:
            assert (end == 0).all()
        assert ((end == 0) | ((end > last) & (end <= T))).all()
    assert (runs[:, 2:6] > 0).any(axis=1).all()


def check_device_tables(T, d):
    """Raises AssertionError where the tables break the kernels' reading of them."""
    tiles, ranges, pairs = d["tiles"], d["ranges"], d["pairs"]
    runs = d["pblk"]
    assert runs.shape[1] == 8
    for ta, tb, b0, cnt in pairs:
        check_runs_as_the_kernels_do(T, runs[b0:b0 + cnt], (True, tb >= 0, False, False))
    # the per-block reading of the runs: {kb, end_a, end_b, causal bits}
    per_pair = [expand_runs(runs[b0:b0 + cnt]) for _, _, b0, cnt in pairs]
    pblk = np.concatenate(per_pair)[:, [0, 1, 2, 5]] if per_pair else np.zeros((0, 4), np.int64)
    pairs = pairs.copy()
    if len(pairs):
        pairs[:, 3] = [len(x) for x in per_pair]
        pairs[:, 2] = np.r_[0, np.cumsum(pairs[:-1, 3])]
    nt = len(tiles)
    assert len(pairs) == (nt + 1) // 2
    begin = 0
    for i, (ta, tb, b0, cnt) in enumerate(pairs):
        assert (ta, tb) == (2 * i, 2 * i + 1 if 2 * i + 1 < nt else -1)
        assert b0 == begin and cnt >= 1
        begin += cnt
    assert begin == len(pblk)
    # the forward kernel's own test of each entry (tile b absent: end_b must be 0)
    tb_of = np.repeat(pairs[:, 1], pairs[:, 3]) if len(pairs) else np.zeros(0, np.int32)
    kb, ea, eb = pblk[:, 0], pblk[:, 1], pblk[:, 2]
    assert ((0 <= kb) & (kb < T) & (ea <= T) & (eb <= T) & ((ea > kb) | (eb > kb))).all()
    assert (((ea == 0) | (ea > kb)) & ((eb == 0) | (eb > kb)) & ((tb_of >= 0) | (eb == 0))).all()
    assert ((tiles[:, 1] >= 0) & (tiles[:, 1] < tiles[:, 2]) & (tiles[:, 2] <= T)).all()
    for ta, tb, b0, cnt in pairs:
        ent = pblk[b0:b0 + cnt]
        assert (np.diff(ent[:, 0]) > 0).all(), "entries not merged by block start"
        for x, t in ((0, ta), (1, tb)):
            if t < 0:
                assert not (ent[:, 3] & 2).any()
                continue
            _, _, _, rb, rc = tiles[t]
            want = [tuple(map(int, ranges[r])) for r in range(rb, rb + rc)]
            last = want[-1]
            end = ent[:, 1 + x]
            causal = ((ent[:, 3] >> x) & 1).astype(bool)
            assert not causal[end == 0].any()
            sel = end > 0
            k0 = ent[sel, 0].astype(np.int64)
            k1 = np.minimum(k0 + BLOCK, end[sel])
            assert (causal[sel] == ((k0 >= last[0]) & (k1 <= last[1]))).all(), "causal flag off the own range"
            assert (k1[:-1] <= k0[1:]).all(), "a key read twice"
            cut = np.nonzero(k1[:-1] != k0[1:])[0]  # merged runs of the covered blocks
            got = list(zip(np.r_[k0[:1], k0[cut + 1]].tolist(), np.r_[k1[cut], k1[-1:]].tolist()))
            assert got == _merge(want), "blocks do not cover the tile's ranges exactly"
    check_quad_tables(T, d)
    bwd, sched = d["bwd"], d["bwd_sched"]
    assert sorted(map(tuple, sched.tolist())) == sorted(map(tuple, bwd.tolist()))
    runs = sched[:, 4] - sched[:, 3]
    assert (np.diff(sched[:, 4]) <= 0).all(), "run ends not latest first"
    for i in range(len(sched) - 1):
        if sched[i, 4] == sched[i + 1, 4]:
            assert runs[i] >= runs[i + 1], "runs of one end not longest first"
            if runs[i] == runs[i + 1]:
                assert sched[i, 1] < sched[i + 1, 1], "ties not in canonical order"
    assert d["run_sum"] == int(runs.sum()) and d["run_max"] == (int(runs.max()) if len(runs) else 0)
    check_merged_blocks(T, d)


def check_merged_blocks(T, d, block=BLOCK):
    """bwd_merged and key_end against the canonical table and the reading above (blocks of
    ``block`` keys)."""
    bwd, rows, key_end = d["bwd"], d["bwd_merged"], d["key_end"]
    want_end = np.zeros(T, dtype=np.int64)
    seg_of = np.zeros(T, dtype=np.int64)
    for seg, k0, k1, q0, q1 in bwd.tolist():
        want_end[k0:k1] = q1
        seg_of[k0:k1] = seg
    assert key_end.shape == (T,) and (key_end == want_end).all(), "a key's run end is off"
    seen = np.zeros(T, dtype=np.int64)
    for seg, k0, k1, q0, q1 in rows.tolist():
        assert 0 <= k0 < k1 <= T and k1 - k0 <= block and q0 == k0, "malformed block"
        assert q1 == key_end[k0] and seg == seg_of[k0], "a block's run is not its first key's"
        assert (key_end[k0:k1] <= q1).all(), "a key seen past its block's run"
        if k1 - k0 < block and k1 < T:
            assert key_end[k1] > q1, "a partial block stops before the end of its subtree's keys"
        seen[k0:k1] += 1
    assert (seen == 1).all(), "keys not covered exactly once"
    runs = rows[:, 4] - rows[:, 3]
    for i in range(len(rows) - 1):
        a, b = rows[i], rows[i + 1]
        assert a[4] > b[4] or (a[4] == b[4] and (runs[i] > runs[i + 1] or (runs[i] == runs[i + 1] and a[1] < b[1]))), \
            "merged blocks not in launch order"
    assert d["runm_sum"] == int(runs.sum()) and d["runm_max"] == (int(runs.max()) if len(runs) else 0)


def _check_entries(tiles, ranges, ent, col, t, bit):
    """Entries of one tile (end in column ``col``, causal flag ``bit``) cover its ranges exactly."""
    _, _, _, rb, rc = tiles[t]
    want = [tuple(map(int, ranges[r])) for r in range(rb, rb + rc)]
    last = want[-1]
    end = ent[:, col]
    causal = ((ent[:, 5] >> bit) & 1).astype(bool)
    assert not causal[end == 0].any()
    sel = end > 0
    k0 = ent[sel, 0].astype(np.int64)
    k1 = np.minimum(k0 + BLOCK, end[sel])
    assert (causal[sel] == ((k0 >= last[0]) & (k1 <= last[1]))).all(), "causal flag off the own range"
    assert (k1[:-1] <= k0[1:]).all(), "a key read twice"
    cut = np.nonzero(k1[:-1] != k0[1:])[0]
    got = list(zip(np.r_[k0[:1], k0[cut + 1]].tolist(), np.r_[k1[cut], k1[-1:]].tolist()))
    assert got == _merge(want), "blocks do not cover the tile's ranges exactly"


def check_quad_tables(T, d):
    """The paired-SM forward's quads and their merged block lists."""
    tiles, ranges, quads = d["tiles"], d["ranges"], d["quads"]
    for a0, a1, b0, b1, e0, cnt in quads:
        check_runs_as_the_kernels_do(T, d["qblk"][e0:e0 + cnt], (a0 >= 0, a1 >= 0, b0 >= 0, b1 >= 0))
    # the per-block reading of the runs: {kb, end a0, a1, b0, b1, causal bits, 0, 0}
    per_quad = [expand_runs(d["qblk"][e0:e0 + cnt]) for *_, e0, cnt in quads]
    qblk = np.concatenate([np.c_[x, np.zeros((len(x), 2), np.int64)] for x in per_quad]) if per_quad \
        else np.zeros((0, 8), np.int64)
    quads = quads.copy()
    if len(quads):
        quads[:, 5] = [len(x) for x in per_quad]
        quads[:, 4] = np.r_[0, np.cumsum(quads[:-1, 5])]
    nt = len(tiles)
    if nt == 0:
        assert len(quads) == 0 and len(qblk) == 0
        return
    seg = tiles[:, 0]
    first = {}
    for t in range(nt):
        first[int(seg[t])] = min(first.get(int(seg[t]), 1 << 40), int(tiles[t, 1]))
    tt = d.get("tile_tokens")
    per_seg = {}
    for t in range(nt):
        per_seg.setdefault(int(seg[t]), []).append(t)
    # tile offset within its segment, from the smallest gap of the segment's tile starts
    offs = np.zeros(nt, np.int64)
    for sg, ts in per_seg.items():
        starts = sorted(int(tiles[t, 1]) for t in ts)
        step = tt or (starts[1] - starts[0] if len(starts) > 1 else 1)
        for t in ts:
            offs[t] = (int(tiles[t, 1]) - first[sg]) // step
    seen = np.zeros(nt, np.int64)
    couples = []
    begin = 0
    for a0, a1, b0, b1, e0, cnt in quads:
        assert a0 >= 0 and e0 == begin and cnt >= 1
        begin += cnt
        for x, y in ((a0, a1), (b0, b1)):
            if x < 0:
                assert y < 0
                continue
            couples.append(x)
            assert offs[x] % 2 == 0, "a couple starts on an odd tile"
            seen[x] += 1
            if y >= 0:
                assert seg[y] == seg[x] and offs[y] == offs[x] + 1, "a couple is not two consecutive tiles"
                seen[y] += 1
            else:
                assert offs[x] == len(per_seg[int(seg[x])]) - 1, "a tile left without its partner"
    assert begin == len(qblk)
    assert (seen == 1).all(), "a tile missing from the quads or in two of them"
    assert couples == sorted(couples), "couples not in schedule order"
    assert (quads[:-1, 2] >= 0).all(), "slot b empty before the last quad"
    present = np.repeat((quads[:, :4] >= 0), quads[:, 5], axis=0)
    kb, ends = qblk[:, 0], qblk[:, 1:5]
    # the paired-SM kernel's own test of each entry
    assert ((0 <= kb) & (kb < T)).all()
    assert (((ends == 0) | (present & (ends > kb[:, None]) & (ends <= T))).all())
    assert (ends > 0).any(axis=1).all()
    assert (qblk[:, 6:] == 0).all()
    for q, (a0, a1, b0, b1, e0, cnt) in enumerate(quads):
        ent = qblk[e0:e0 + cnt]
        assert (np.diff(ent[:, 0]) > 0).all(), "entries not merged by block start"
        for i, t in enumerate((a0, a1, b0, b1)):
            if t < 0:
                assert not (ent[:, 1 + i]).any() and not ((ent[:, 5] >> i) & 1).any()
                continue
            _check_entries(tiles, ranges, ent, 1 + i, t, i)


def random_run_lists(rng, block=BLOCK):
    """Up to four slots of sorted, disjoint ranges with arbitrary starts (aligned or not with each other)."""
    lists = []
    for _ in range(4):
        if rng.random() < 0.2:
            lists.append([])
            continue
        pos, runs = int(rng.integers(0, 300)), []
        for r in range(int(rng.integers(1, 5))):
            a = pos + int(rng.integers(0, 3)) * int(rng.choice([block, 37, 64]))
            e = a + int(rng.integers(1, 5 * block))
            runs.append((a, -(-(e - a) // block), e, int(r == 0)))
            pos = e
        lists.append(runs)
    return lists


def check_run_merge(host, lists, block=BLOCK):
    """The planner's run merge, expanded block by block, equals a merge of the slots' blocks by start."""
    got = expand_runs(host.merge_runs(lists, block)) if any(lists) else np.zeros((0, 6), np.int64)
    want = {}
    for i, runs in enumerate(lists):
        for a, nb, e, causal in runs:
            for k in range(nb):
                row = want.setdefault(a + block * k, [a + block * k, 0, 0, 0, 0, 0])
                row[1 + i] = e
                row[5] |= causal << i
    assert got.tolist() == [want[k] for k in sorted(want)]


def test_run_merge_equals_a_block_by_block_merge(host):
    rng = np.random.default_rng(23)
    for _ in range(300):
        check_run_merge(host, random_run_lists(rng))


@pytest.fixture(scope="module")
def host(tmp_path_factory):
    d = tmp_path_factory.mktemp("device_tables")
    return build_host_library(original_objects(d), d / "lib")


def _tables(host, t, tile, order=0):
    d = host.device_tables(t.seg_start, t.seg_len, t.parent, t.depth, tile, BLOCK, order)
    assert not isinstance(d, int), f"refused ({d})"
    d["tile_tokens"] = tile
    return d


@pytest.mark.parametrize("name", ["tiny", "star", "agent", "forest", "long"])
@pytest.mark.parametrize("order", [0, 1])
def test_workload_tables(host, name, order):
    w = W.get(name)
    check_device_tables(w.T, _tables(host, w.tree, 128 // (w.hq // w.hkv), order))


def test_random_tree_tables(host):
    rng = np.random.default_rng(8)
    for _ in range(80):
        t = W.random_small_tree(rng, max_segments=12, max_len=400)
        check_device_tables(t.total_tokens, _tables(host, t, int(rng.choice([16, 32, 64, 128])),
                                                     int(rng.integers(0, 2))))


def test_single_tile_and_empty_plans(host):
    one = W.tree_from_preorder([40], [-1])
    d = _tables(host, one, 128)
    assert d["pairs"].tolist() == [[0, -1, 0, 1]] and d["pblk"].tolist() == [[0, 1, 40, 0, 0, 0, 1, 0]]
    assert d["quads"].tolist() == [[0, -1, -1, -1, 0, 1]] and d["qblk"].tolist() == [[0, 1, 40, 0, 0, 0, 1, 0]]
    check_device_tables(40, d)
    empty = host.device_tables([], [], [], [], 128, BLOCK, 0)
    assert len(empty["pairs"]) == 0 and len(empty["bwd_sched"]) == 0 and empty["run_max"] == 0


def test_the_checks_catch_broken_tables(host):
    t = W.tiny().tree
    good = _tables(host, t, 32)
    check_device_tables(t.total_tokens, good)
    breaks = [
        lambda d: d["pblk"].__setitem__((0, 6), d["pblk"][0, 6] ^ 1),        # a causal bit flipped
        lambda d: d["pblk"].__setitem__((0, 2), d["pblk"][0, 2] - 1),        # a block end cut short
        lambda d: d["pblk"].__setitem__((0, 1), d["pblk"][0, 1] + 1),        # a run one block too long
        lambda d: d["pairs"].__setitem__((0, 3), d["pairs"][0, 3] - 1),      # a run dropped from a pair
        lambda d: d["bwd_sched"].__setitem__(slice(None), d["bwd_sched"][::-1].copy()),  # launch order reversed
        lambda d: d.__setitem__("run_max", d["run_max"] + 1),
    ]
    breaks += [
        lambda d: d["qblk"].__setitem__((0, 6), d["qblk"][0, 6] ^ 1),        # a quad's causal bit flipped
        lambda d: d["qblk"].__setitem__((0, 2), d["qblk"][0, 2] - 1),        # a quad's block end cut short
        lambda d: d["quads"].__setitem__((0, 5), d["quads"][0, 5] - 1),      # a run dropped from a quad
        lambda d: d["quads"].__setitem__((0, 1), d["quads"][0, 2]),          # a couple of two segments
        lambda d: d["key_end"].__setitem__(0, d["key_end"][0] + 1),          # a key's run end off by one
        lambda d: d["bwd_merged"].__setitem__((0, 4), d["bwd_merged"][0, 4] - 1),  # a block's run cut short
        lambda d: d["bwd_merged"].__setitem__(slice(None), d["bwd_merged"][::-1].copy()),  # order reversed
        lambda d: d.__setitem__("runm_sum", d["runm_sum"] + 1),
        lambda d: d.__setitem__("bwd_merged", d["bwd_sched"].copy()),       # partial blocks left unfilled
    ]
    for brk in breaks:
        bad = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in good.items()}
        brk(bad)
        with pytest.raises(AssertionError):
            check_device_tables(t.total_tokens, bad)
