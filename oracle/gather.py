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
