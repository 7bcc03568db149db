"""Independent planner for the per-query-tile ancestor KV ranges (oracle).

Issue #7386 ("Describe the solution you'd like", third bullet): each query
run attends to its ancestor path only; PR #7387 ("Summary", second bullet): a
query segment attends causally over its ancestors.  A plan lists, for every query tile, the key ranges that tile
reads: the ancestor segments' tokens (fully visible) and the own segment up to
the tile's end (causal).  The pages fix no tile size or order; the canonical
form below is this library's, and the C++ planner must reproduce it bit for
bit.

Canonical form, for ``tile_tokens`` (query tokens per tile) and ``kv_block``
(keys per backward block):

* tiles: every segment is cut from its start into tiles of ``tile_tokens``
  tokens; the last tile of a segment may be shorter; no tile crosses a
  segment end.
* ranges of a tile: the token intervals of the strict ancestors, root first,
  then ``[seg_start, q_end)``; touching intervals (end == next start) are
  merged.  The last range of a tile is the causal one (key j visible to query
  i iff j <= i); all earlier ranges are fully visible.
* tile order 0 ("siblings adjacent"): ascending (root segment, parent segment
  or -1, tile index inside the segment, segment); order 1 ("longest first"):
  descending total range length, then segment, then tile index.
* backward table: every segment is cut into blocks of ``kv_block`` keys; each
  block reads the queries ``[kv_start, end of the segment's subtree)``; blocks
  come in descending query-count order, ties by ``kv_start``.

This module walks parent pointers for every tile and sorts with Python tuple
keys; it deliberately does not mirror the C++ planner's single stack pass.
"""
from __future__ import annotations

import numpy as np

from . import tree as _tree


def _root_of(parent, s):
    while int(parent[s]) != -1:
        s = int(parent[s])
    return s


def _merge(intervals):
    out = []
    for a, b in sorted(intervals):
        if out and out[-1][1] == a:
            out[-1] = (out[-1][0], b)
        else:
            out.append((a, b))
    return out


def subtree_end(seg_start, seg_len, parent, s) -> int:
    """One past the last token of any segment in s's subtree."""
    return max(int(seg_start[d]) + int(seg_len[d]) for d in _tree.descendants(parent, s))


def build(seg_start, seg_len, parent, tile_tokens: int, kv_block: int, order: int = 0):
    """Return (tiles [n,5], ranges [m,2], bwd [k,5]) as int32 arrays.

    tiles rows: (seg, q_start, q_end, r_begin, r_count); ranges rows:
    (kv_start, kv_end); bwd rows: (seg, kv_start, kv_end, q_begin, q_end).
    """
    n = len(seg_len)
    raw = []  # (sort_key, seg, q_start, q_end, ranges)
    for s in range(n):
        a0 = int(seg_start[s])
        a1 = a0 + int(seg_len[s])
        anc = _tree.ancestors(parent, s)
        anc_iv = [(int(seg_start[a]), int(seg_start[a]) + int(seg_len[a])) for a in anc]
        k = 0
        for q0 in range(a0, a1, tile_tokens):
            q1 = min(q0 + tile_tokens, a1)
            rng = _merge(anc_iv + [(a0, q1)])
            if order == 0:
                key = (_root_of(parent, s), int(parent[s]), k, s)
            else:
                key = (-sum(b - a for a, b in rng), s, k)
            raw.append((key, s, q0, q1, rng))
            k += 1
    raw.sort(key=lambda r: r[0])
    tiles, ranges = [], []
    for _, s, q0, q1, rng in raw:
        tiles.append((s, q0, q1, len(ranges), len(rng)))
        ranges.extend(rng)

    bwd = []
    for s in range(n):
        a0 = int(seg_start[s])
        a1 = a0 + int(seg_len[s])
        qe = subtree_end(seg_start, seg_len, parent, s)
        for k0 in range(a0, a1, kv_block):
            bwd.append((s, k0, min(k0 + kv_block, a1), k0, qe))
    bwd.sort(key=lambda r: (-(r[4] - r[3]), r[1]))

    as32 = lambda x, w: np.asarray(x, dtype=np.int32).reshape(-1, w)  # noqa: E731
    return as32(tiles, 5), as32(ranges, 2), as32(bwd, 5)


def expand_forward_mask(T, tiles, ranges) -> np.ndarray:
    """Boolean T x T mask implied by a forward plan (for checking plans)."""
    m = np.zeros((T, T), dtype=bool)
    for s, q0, q1, rb, rc in tiles:
        for r in range(rb, rb + rc):
            k0, k1 = ranges[r]
            for i in range(q0, q1):
                for j in range(k0, k1):
                    if r < rb + rc - 1 or j <= i:
                        m[i, j] = True
    return m


def expand_backward_mask(T, bwd) -> np.ndarray:
    """Boolean T x T mask implied by the backward table (for checking plans)."""
    m = np.zeros((T, T), dtype=bool)
    for s, k0, k1, q0, q1 in bwd:
        for j in range(k0, k1):
            for i in range(q0, q1):
                if j <= i:
                    m[i, j] = True
    return m
