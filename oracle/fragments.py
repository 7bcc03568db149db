"""Bounded fragment planning (oracle).

"[ENHANCEMENT] Shared-prefix training with context parallelism for exact
agent trajectories" (issue #7386), "Describe the solution you'd like" (third
and last paragraphs): the trainer keeps fragments under a memory limit, with
ancestors repeated in several fragments where needed, and every sampled action
keeps exactly one loss owner ("Additional context": 3,744,651 physical tokens before
fragment duplication, 3,919,929 after).  The pages give no algorithm; the
reading implemented here, in plain Python:

* A fragment is a set of segments closed under "parent of", so every segment
  in it comes with its whole root path, and its physical tokens (the sum of
  its segments' lengths) are at most ``max_tokens``.
* Segments are visited in preorder.  Segment s joins the current fragment
  together with whichever of its ancestors the fragment lacks, if that keeps
  the fragment within the cap; otherwise the current fragment is closed and a
  new one starts from s's root path.
* The fragment that takes s in its own visit owns s (its tokens' loss and
  outputs); ancestors brought in again are context only.  Each segment is
  therefore owned exactly once.
* A root path longer than the cap cannot be placed: ValueError.

Test infrastructure only.
"""
from __future__ import annotations

import numpy as np


def plan_fragments(seg_len, parent, max_tokens: int):
    """Returns a list of fragments; each is a list of (segment, owned) in preorder."""
    seg_len = [int(x) for x in seg_len]
    parent = [int(p) for p in parent]
    n = len(seg_len)
    frags = []
    cur, cur_set, cur_tokens = [], set(), 0
    for s in range(n):
        path = []
        a = s
        while a >= 0:
            path.append(a)
            a = parent[a]
        path.reverse()  # root first
        path_tokens = sum(seg_len[a] for a in path)
        if path_tokens > max_tokens:
            raise ValueError(f"root path of segment {s} has {path_tokens} tokens, above the cap {max_tokens}")
        missing = [a for a in path if a not in cur_set]
        extra = sum(seg_len[a] for a in missing)
        if cur and cur_tokens + extra > max_tokens:
            frags.append(cur)
            cur, cur_set, cur_tokens = [], set(), 0
            missing, extra = path, path_tokens
        for a in missing:
            cur.append((a, a == s))
            cur_set.add(a)
        cur_tokens += extra
    if cur:
        frags.append(cur)
    # preorder within each fragment (segment ids are preorder positions)
    return [sorted(f) for f in frags]


def fragment_tokens(frags, seg_len) -> int:
    return int(sum(int(seg_len[a]) for f in frags for a, _ in f))


def check_fragments(frags, seg_len, parent, max_tokens: int) -> None:
    """Raises AssertionError unless the fragments are a valid bounded cover."""
    n = len(seg_len)
    owners = np.zeros(n, dtype=np.int64)
    for f in frags:
        segs = [a for a, _ in f]
        assert segs == sorted(set(segs)), "fragment not in preorder or with repeats"
        present = set(segs)
        assert sum(int(seg_len[a]) for a in segs) <= max_tokens, "fragment above the cap"
        for a, owned in f:
            if parent[a] >= 0:
                assert int(parent[a]) in present, "fragment not closed under parent"
            if owned:
                owners[a] += 1
    assert (owners == 1).all(), "a segment is not owned exactly once"
