"""Log-probability of each sampled action through the vocabulary head (oracle).

Issue #7386 ("Describe the solution you'd like", fifth bullet): only the hidden
states at sampled-edge source tokens go through the vocabulary projection, and
every sampled action keeps exactly one loss owner.  PR #7387 ("Summary",
fourth bullet) selects those states before the projection.

The pages name neither the loss nor the vocabulary size.  Reading used here:
the quantity each action owns is the log-probability of its sampled token,

    logits[e, v] = <hidden_sel[e], weight[v]>
    lse[e]       = log sum_v exp(logits[e, v])
    logprob[e]   = logits[e, labels[e]] - lse[e]

(weight is [V, Hd], the layout of a linear layer's weight), and its backward
for an upstream gradient g[e] = dL/dlogprob[e]:

    dlogits[e, v]  = g[e] * (1[v == labels[e]] - exp(logits[e, v] - lse[e]))
    d_hidden_sel   = dlogits @ weight
    d_weight       = dlogits^T @ hidden_sel

Everything in fp64.  Test infrastructure only.
"""
from __future__ import annotations

import numpy as np


def _check(hidden_sel, weight, labels):
    hidden_sel = np.asarray(hidden_sel, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    labels = np.asarray(labels, dtype=np.int64)
    E, Hd = hidden_sel.shape
    V, Hd2 = weight.shape
    if Hd != Hd2 or labels.shape != (E,):
        raise ValueError("shape mismatch")
    if E and (labels.min() < 0 or labels.max() >= V):
        raise IndexError("label outside the vocabulary")
    return hidden_sel, weight, labels


def logits(hidden_sel, weight) -> np.ndarray:
    """[E, V] projection of the selected states (a plain matrix product)."""
    return np.asarray(hidden_sel, dtype=np.float64) @ np.asarray(weight, dtype=np.float64).T


def log_sum_exp_rows(z: np.ndarray) -> np.ndarray:
    """log sum_v exp(z[e, v]) per row, shifted by the row maximum so that it cannot overflow."""
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def edge_logprob(hidden_sel, weight, labels):
    """Returns (logprob[E], lse[E]) for the sampled labels."""
    hidden_sel, weight, labels = _check(hidden_sel, weight, labels)
    if hidden_sel.shape[0] == 0:
        return np.zeros(0), np.zeros(0)
    z = logits(hidden_sel, weight)
    lse = log_sum_exp_rows(z)
    return z[np.arange(len(labels)), labels] - lse, lse


def edge_logprob_backward(hidden_sel, weight, labels, grad_logprob):
    """Returns (d_hidden_sel [E, Hd], d_weight [V, Hd]) for upstream grad_logprob[E]."""
    hidden_sel, weight, labels = _check(hidden_sel, weight, labels)
    g = np.asarray(grad_logprob, dtype=np.float64)
    E = hidden_sel.shape[0]
    if E == 0:
        return np.zeros_like(hidden_sel), np.zeros_like(weight)
    z = logits(hidden_sel, weight)
    p = np.exp(z - log_sum_exp_rows(z)[:, None])
    dz = -p
    dz[np.arange(E), labels] += 1.0
    dz *= g[:, None]
    return dz @ weight, dz.T @ hidden_sel


def weight_grad_rows(hidden_sel, weight, labels, grad_logprob, vocab_rows):
    """Rows ``vocab_rows`` of ``edge_logprob_backward``'s d_weight.

    The same definition, evaluated only for the requested vocabulary rows:
    the softmax still normalises over the whole vocabulary (the [E, V] logits
    are formed in full), only the columns of dlogits that those rows need are
    built.  For checking a large d_weight one row at a time.
    """
    hidden_sel, weight, labels = _check(hidden_sel, weight, labels)
    g = np.asarray(grad_logprob, dtype=np.float64)
    rows = np.asarray(vocab_rows, dtype=np.int64)
    z = logits(hidden_sel, weight)
    lse = log_sum_exp_rows(z)
    dz = -np.exp(z[:, rows] - lse[:, None])
    dz += (labels[:, None] == rows[None, :])
    dz *= g[:, None]
    return dz.T @ hidden_sel
