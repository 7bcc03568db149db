"""Shared-prefix tree attention, forward and backward, in fp64 (oracle).

What is computed.  Issue #7386 ("Describe alternatives you've considered",
item 1) names independent exact-call sequences as the correctness reference:
every root-to-leaf call is an ordinary causal sequence.  The tree result must
equal that reference while each shared prefix is stored once.  So the forward
here unrolls each root-to-leaf path into its own sequence, runs plain causal
softmax attention on it and maps every row back to its physical token; a
prefix token that lies on several paths must come out the same on all of them
(checked).

Backward.  #7914 (introduction): the backward sums every branch's
contribution into the prefix the branches share.  The loss of the tree is
``L = sum_i <O_i, dO_i>`` over physical tokens.  In the unrolled sequences
each physical token's upstream gradient dO is handed to exactly one copy --
the first root-to-leaf path in DFS order that contains it -- and all other
copies get zero; this is the pages' rule that each sampled action has a
single loss owner (issue #7386, "Describe the solution you'd like", fifth bullet, and
"Additional context") applied to the upstream gradient, and it is the only
assignment for which the unrolled sum equals dL of the tree.  Per path the
gradient is the textbook one (dV = P^T dO, dP = dO V^T, D = rowsum(dO*O),
dS = P*(dP - D), dQ = scale dS K, dK = scale dS^T Q); the per-path results
are scatter-added onto the physical tokens, which sums prefix gradients over
branches.

Conventions (the pages are silent): softmax scale is an argument; LSE is the
natural log of the row's sum of exp(scale * q.k), stored ``[Hq, T]``; query
head h reads KV head ``h // (Hq // Hkv)``.

Arrays: q, do ``[T, Hq, D]``; k, v ``[T, Hkv, D]``; any float dtype (bf16
values should be passed as float32 or float64, which hold them exactly); all
arithmetic is float64.
"""
from __future__ import annotations

import numpy as np

from . import tree as _tree

ROW_CHUNK = 1024


def causal_rows(qp, kp, vp, rows, scale, dop=None):
    """Plain causal attention for selected rows of one ordinary sequence.

    qp, kp, vp (and dop): ``[n, D]`` float64.  ``rows``: ascending positions.
    Row r attends to keys 0..r.  Returns (O[rows], LSE[rows]) and, when dop is
    given, also (dQ[rows], dK[n], dV[n]) for the loss sum_r <O_r, dop_r> over
    the selected rows only.
    """
    rows = np.asarray(rows, dtype=np.int64)
    n, D = kp.shape
    O = np.empty((len(rows), D))
    LSE = np.empty(len(rows))
    grads = dop is not None
    if grads:
        dQ = np.empty((len(rows), D))
        dK = np.zeros((n, D))
        dV = np.zeros((n, D))
    for c0 in range(0, len(rows), ROW_CHUNK):
        r = rows[c0:c0 + ROW_CHUNK]
        kmax = int(r[-1]) + 1
        S = scale * (qp[r] @ kp[:kmax].T)
        S[np.arange(kmax)[None, :] > r[:, None]] = -np.inf
        m = S.max(axis=1)
        P = np.exp(S - m[:, None])
        l = P.sum(axis=1)
        P /= l[:, None]
        Oc = P @ vp[:kmax]
        O[c0:c0 + len(r)] = Oc
        LSE[c0:c0 + len(r)] = m + np.log(l)
        if grads:
            dOc = dop[r]
            Dv = (dOc * Oc).sum(axis=1)
            dP = dOc @ vp[:kmax].T
            dS = P * (dP - Dv[:, None])
            dQ[c0:c0 + len(r)] = scale * (dS @ kp[:kmax])
            dK[:kmax] += scale * (dS.T @ qp[r])
            dV[:kmax] += P.T @ dOc
    if grads:
        return O, LSE, dQ, dK, dV
    return O, LSE


def _groups(hq, hkv, groups):
    G = hq // hkv
    gs = range(hkv) if groups is None else groups
    return G, [int(g) for g in gs]


def path_attention(q, k, v, scale, path_idx, group, rows=None, do=None):
    """One root-to-leaf call unrolled as an ordinary causal sequence.

    ``path_idx``: the call's physical token indices in order.  ``group``: the
    KV head whose G query heads are computed.  ``rows``: positions (within
    the path) whose outputs are formed and whose dO enters the loss; default
    all.  Returns a dict with ``O`` [len(rows), G, D], ``LSE`` [G, len(rows)]
    and, with ``do``, ``dQ`` [len(rows), G, D] plus ``dK``/``dV`` [n, D]
    summed over the G query heads.
    """
    hq, hkv = q.shape[1], k.shape[1]
    G = hq // hkv
    idx = np.asarray(path_idx, dtype=np.int64)
    n = len(idx)
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    kp = np.asarray(k[idx, group, :], dtype=np.float64)
    vp = np.asarray(v[idx, group, :], dtype=np.float64)
    D = kp.shape[1]
    out = {"O": np.empty((len(rows), G, D)), "LSE": np.empty((G, len(rows)))}
    if do is not None:
        out["dQ"] = np.empty((len(rows), G, D))
        out["dK"] = np.zeros((n, D))
        out["dV"] = np.zeros((n, D))
    if len(rows) == 0:
        return out
    for j in range(G):
        h = group * G + j
        qp = np.asarray(q[idx, h, :], dtype=np.float64)
        if do is None:
            O, L = causal_rows(qp, kp, vp, rows, scale)
        else:
            dop = np.asarray(do[idx, h, :], dtype=np.float64)
            O, L, dQ, dK, dV = causal_rows(qp, kp, vp, rows, scale, dop)
            out["dQ"][:, j] = dQ
            out["dK"] += dK
            out["dV"] += dV
        out["O"][:, j] = O
        out["LSE"][j] = L
    return out


def tree_forward(q, k, v, seg_start, seg_len, parent, scale, groups=None, check_tol=1e-12):
    """O [T, Hq, D] and LSE [Hq, T] by unrolling every root-to-leaf path.

    Only the query heads of the KV groups in ``groups`` (default all) are
    filled; other entries stay NaN.
    """
    T, hq, D = q.shape
    hkv = k.shape[1]
    G, gs = _groups(hq, hkv, groups)
    O = np.full((T, hq, D), np.nan)
    LSE = np.full((hq, T), np.nan)
    for g in gs:
        hs = slice(g * G, (g + 1) * G)
        seen = np.zeros(T, dtype=bool)
        for leaf in _tree.leaves(parent):
            idx = _tree.path_tokens(seg_start, seg_len, parent, leaf)
            r = path_attention(q, k, v, scale, idx, g)
            old = seen[idx]
            if old.any():
                prev = O[idx[old], hs]
                err = np.abs(r["O"][old] - prev).max() / max(np.abs(prev).max(), 1e-300)
                if err > check_tol:
                    raise AssertionError(f"prefix outputs differ between paths by {err:.3e}")
            new = ~old
            O[idx[new], hs] = r["O"][new]
            LSE[hs, idx[new]] = r["LSE"][:, new]
            seen[idx] = True
    return O, LSE


def tree_backward(q, k, v, do, seg_start, seg_len, parent, scale, groups=None, owner="first"):
    """dQ [T,Hq,D], dK [T,Hkv,D], dV [T,Hkv,D] of L = sum_i <O_i, dO_i>.

    Each physical token's dO is owned by the first (``owner='first'``) or the
    last (``owner='last'``) root-to-leaf path in DFS order that contains it.
    """
    T, hq, D = q.shape
    hkv = k.shape[1]
    G, gs = _groups(hq, hkv, groups)
    dQ = np.full((T, hq, D), np.nan)
    dK = np.full((T, hkv, D), np.nan)
    dV = np.full((T, hkv, D), np.nan)
    order = _tree.leaves(parent)
    if owner == "last":
        order = order[::-1]
    for g in gs:
        hs = slice(g * G, (g + 1) * G)
        dQ[:, hs] = 0.0
        dK[:, g] = 0.0
        dV[:, g] = 0.0
        seen = np.zeros(T, dtype=bool)
        for leaf in order:
            idx = _tree.path_tokens(seg_start, seg_len, parent, leaf)
            own = np.nonzero(~seen[idx])[0]
            seen[idx] = True
            if len(own) == 0:
                continue
            r = path_attention(q, k, v, scale, idx, g, rows=own, do=do)
            dQ[idx[own], hs] += r["dQ"]
            np.add.at(dK[:, g], idx, r["dK"])
            np.add.at(dV[:, g], idx, r["dV"])
    return dQ, dK, dV


def dense_forward(q, k, v, mask, scale):
    """Second route for tiny trees: masked softmax attention over all T keys.

    ``mask``: T x T boolean visibility (from the brute-force parent walk).
    Returns O [T, Hq, D], LSE [Hq, T], and P [Hq, T, T].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, hq, D = q.shape
    G = hq // k.shape[1]
    O = np.empty_like(q)
    LSE = np.empty((hq, T))
    P = np.empty((hq, T, T))
    for h in range(hq):
        S = scale * (q[:, h] @ k[:, h // G].T)
        S = np.where(mask, S, -np.inf)
        m = S.max(axis=1)
        E = np.exp(S - m[:, None])
        l = E.sum(axis=1)
        P[h] = E / l[:, None]
        O[:, h] = P[h] @ v[:, h // G]
        LSE[h] = m + np.log(l)
    return O, LSE, P


def dense_backward(q, k, v, do, mask, scale):
    """Gradient of sum_i <O_i, dO_i> through ``dense_forward``."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    T, hq, D = q.shape
    hkv = k.shape[1]
    G = hq // hkv
    O, _, P = dense_forward(q, k, v, mask, scale)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    for h in range(hq):
        g = h // G
        dV[:, g] += P[h].T @ do[:, h]
        dP = do[:, h] @ v[:, g].T
        Dv = (do[:, h] * O[:, h]).sum(axis=1)
        dS = P[h] * (dP - Dv[:, None])
        dQ[:, h] = scale * (dS @ k[:, g])
        dK[:, g] += scale * (dS.T @ q[:, h])
    return dQ, dK, dV


def subtree_key_grads(q, k, v, do, seg_start, seg_len, parent, scale, seg, group):
    """dK, dV [len(seg), D] of segment ``seg``'s keys for KV head ``group``.

    Only queries in seg's subtree can see seg's keys, so this is
    ``tree_backward`` restricted to the root-to-leaf paths through ``seg``:
    each physical token of the subtree is owned by the first such path (DFS
    order) that contains it.  Cost grows with the subtree, not the tree.
    """
    sub = set(_tree.descendants(parent, seg))
    a0, a1 = int(seg_start[seg]), int(seg_start[seg]) + int(seg_len[seg])
    D = k.shape[2]
    dK = np.zeros((a1 - a0, D))
    dV = np.zeros((a1 - a0, D))
    seen = set()
    for leaf in _tree.leaves(parent):
        if leaf not in sub:
            continue
        idx = _tree.path_tokens(seg_start, seg_len, parent, leaf)
        inside = (idx >= a0)  # tokens of seg and below on this path
        own = np.array([p for p in np.nonzero(inside)[0] if int(idx[p]) not in seen], dtype=np.int64)
        seen.update(int(t) for t in idx[inside])
        if len(own) == 0:
            continue
        r = path_attention(q, k, v, scale, idx, group, rows=own, do=do)
        pos = np.nonzero((idx >= a0) & (idx < a1))[0]
        dK += r["dK"][pos]
        dV += r["dV"][pos]
    return dK, dV
