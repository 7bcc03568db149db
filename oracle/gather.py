"""Sampled-edge source selection (oracle).

Issue #7386 ("Describe the solution you'd like", fifth bullet) and PR #7387
("Summary", fourth bullet): only the hidden states at sampled-edge source
indices go through the vocabulary projection.  The selection itself is a row
gather; duplicate indices are legal (several child branches may share one
source token, and each sampled action keeps its own row).
"""
from __future__ import annotations

import numpy as np


def edge_gather(hidden: np.ndarray, idx) -> np.ndarray:
    """``out[e] = hidden[idx[e]]``; raises IndexError on an index outside [0, T)."""
    idx = np.asarray(idx, dtype=np.int64)
    T = hidden.shape[0]
    if idx.size and (idx.min() < 0 or idx.max() >= T):
        raise IndexError("edge index outside the token range")
    return hidden[idx]


def edge_gather_backward(grad_out: np.ndarray, idx, num_tokens: int) -> np.ndarray:
    """Gradient of ``edge_gather`` with respect to ``hidden``.

    Each sampled action's row of upstream gradient flows back to its source
    token; a token that is the source of several actions (a branch point
    shared by several child calls) receives the sum of their rows.  Rows of
    tokens that are no action's source are zero.  Summation order: ascending
    action index (fixes the rounding of a sum in lower precision).
    """
    idx = np.asarray(idx, dtype=np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= num_tokens):
        raise IndexError("edge index outside the token range")
    out = np.zeros((num_tokens,) + grad_out.shape[1:], dtype=np.float64)
    for e in range(len(idx)):  # plain loop: one row per sampled action, in order
        out[idx[e]] += grad_out[e]
    return out
