"""Tree metadata: validation, ancestry and brute-force visibility (oracle).

A tree is four int arrays over segments in DFS preorder: ``seg_start``,
``seg_len``, ``parent`` (-1 for a root) and ``depth``.  Issue #7386 ("Describe
the solution you'd like", first bullet) and PR #7387 ("Summary", first bullet)
describe this metadata as DFS-linearized segments with parent/depth
(ancestor) information.  Reading taken: "DFS-linearized" is preorder, the one
DFS order in which every ancestor precedes its descendants, which a query
segment attending causally over its ancestors (PR #7387, "Summary") needs.

Rejection of malformed input before any work follows #7914 (introduction:
unsupported layouts and modes are refused before anything runs) and PR #7387
("Summary": unsupported input is rejected).
"""
from __future__ import annotations

import numpy as np


class InvalidTree(ValueError):
    pass


def validate(seg_start, seg_len, parent, depth, total_tokens=None) -> None:
    """Raise InvalidTree unless the arrays describe a packed preorder forest.

    Checks, in order: equal lengths; dense packing from token 0 with every
    segment non-empty; parent index before the child (or -1); depth equal to
    the parent's depth + 1 (0 at a root); and preorder contiguity, i.e. each
    segment's parent lies on the root path of the previously placed segment.
    """
    seg_start = [int(x) for x in seg_start]
    seg_len = [int(x) for x in seg_len]
    parent = [int(x) for x in parent]
    depth = [int(x) for x in depth]
    n = len(seg_len)
    if not (len(seg_start) == len(parent) == len(depth) == n):
        raise InvalidTree("array lengths differ")
    pos = 0
    for s in range(n):
        if seg_len[s] < 1:
            raise InvalidTree(f"segment {s} is empty")
        if seg_start[s] != pos:
            raise InvalidTree(f"segment {s} does not start where segment {s - 1} ends")
        pos += seg_len[s]
    if total_tokens is not None and pos != int(total_tokens):
        raise InvalidTree("segment lengths do not add up to the token count")
    if n and parent[0] != -1:
        raise InvalidTree("the first segment must be a root")
    for s in range(n):
        p = parent[s]
        if p < -1 or p >= s:
            raise InvalidTree(f"segment {s} has parent {p}, not an earlier segment")
        want = 0 if p == -1 else depth[p] + 1
        if depth[s] != want:
            raise InvalidTree(f"segment {s} has depth {depth[s]}, expected {want}")
    # the root path of the last placed segment, rebuilt by walking parents
    last = None
    for s in range(n):
        p = parent[s]
        if p != -1:
            on_path = set()
            a = last
            while a is not None and a != -1:
                on_path.add(a)
                a = parent[a]
            if p not in on_path:
                raise InvalidTree(f"segment {s} is not in DFS preorder (parent {p} closed)")
        last = s


def segment_of_token(seg_start, seg_len) -> np.ndarray:
    """seg(i) for every token i."""
    return np.repeat(np.arange(len(seg_len)), np.asarray(seg_len, dtype=np.int64))


def ancestors(parent, s) -> list[int]:
    """Strict ancestors of segment s, root first (a parent-pointer walk)."""
    out = []
    a = int(parent[s])
    while a != -1:
        out.append(a)
        a = int(parent[a])
    return out[::-1]


def children(parent) -> list[list[int]]:
    ch: list[list[int]] = [[] for _ in range(len(parent))]
    for s, p in enumerate(parent):
        if p >= 0:
            ch[int(p)].append(s)
    return ch


def leaves(parent) -> list[int]:
    """Segments with no child, in preorder (= DFS order of leaves)."""
    ch = children(parent)
    return [s for s in range(len(parent)) if not ch[s]]


def path_tokens(seg_start, seg_len, parent, leaf) -> np.ndarray:
    """Token indices of the root-to-leaf call ending at segment ``leaf``."""
    segs = ancestors(parent, leaf) + [leaf]
    return np.concatenate([np.arange(int(seg_start[a]), int(seg_start[a]) + int(seg_len[a])) for a in segs])


def descendants(parent, s) -> list[int]:
    """Segment s and everything below it (by walking the children lists)."""
    ch = children(parent)
    out, todo = [], [s]
    while todo:
        a = todo.pop()
        out.append(a)
        todo.extend(ch[a])
    return sorted(out)


def visible_mask_bruteforce(seg_start, seg_len, parent) -> np.ndarray:
    """T x T boolean: query token i may attend to key token j.

    Straight from the rule on the pages: j is visible to i iff seg(j) is a
    strict ancestor of seg(i) (full attention to the ancestor path), or
    seg(j) == seg(i) and j <= i (causal inside the query's own segment).
    Every (i, j) pair is decided by its own parent walk.
    """
    seg = segment_of_token(seg_start, seg_len)
    T = len(seg)
    m = np.zeros((T, T), dtype=bool)
    for i in range(T):
        anc = set(ancestors(parent, int(seg[i])))
        for j in range(T):
            if seg[j] == seg[i]:
                m[i, j] = j <= i
            else:
                m[i, j] = int(seg[j]) in anc
    return m
