"""Vocabulary head over the sampled-edge states: CUDA path vs the fp64 oracle.

Tolerance: logits accumulate Hd bf16 products in fp32 (relative error about
Hd * 2^-24 of sum |h_d w_d|, below 1e-6 here), the tile sums use ex2.approx
(relative error about 2^-22 per term) and fp32 sums over V terms; lse and
logprob therefore agree with the fp64 oracle to well under 1e-4 absolute,
the bound the tests use.
"""
import numpy as np
import pytest
import torch

import shared_prefix_causal_gb300 as spc
import workloads as W
from oracle import lm_head as LH

pytestmark = pytest.mark.gpu
TOL = 1e-4


def _run(h, w, y):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp, lse = spc.edge_logprob(h.cuda(), w.cuda(), y.cuda(), st)
    torch.cuda.synchronize()
    return lp.cpu(), lse.cpu(), st.item()


@pytest.mark.parametrize("E,V,Hd", [(1, 1, 8), (5, 300, 64), (300, 1000, 200), (129, 513, 136), (260, 4096, 512)])
def test_edge_logprob_matches_oracle(E, V, Hd):
    x = W.draw_lm_head(E, Hd, V, seed=E + V)
    h, w, y = x["hidden_sel"], x["weight"], x["labels"]
    # labels on tile edges where the vocabulary allows it
    edge = torch.tensor([0, 255, 256, V - 1, 511, 512], dtype=torch.int32)
    y[: min(E, 6)] = torch.clamp(edge[: min(E, 6)], max=V - 1)
    lp, lse, st = _run(h, w, y)
    assert st == 0
    rlp, rlse = LH.edge_logprob(h.double().numpy(), w.double().numpy(), y.numpy())
    assert np.abs(lse.double().numpy() - rlse).max() <= TOL
    assert np.abs(lp.double().numpy() - rlp).max() <= TOL


def test_edge_logprob_full_size_sampled_rows():
    """Agent-tree action count, hidden 4096, vocabulary 131,072: the bench's launch, rows checked one by one."""
    w = W.get("agent")
    E = len(w.edge_idx)
    x = W.draw_lm_head(E, w.hidden_dim, seed=3)
    h, wt, y = x["hidden_sel"], x["weight"], x["labels"]
    lp, lse, st = _run(h, wt, y)
    assert st == 0
    rows = np.unique(np.concatenate([[0, 1, 127, 128, E - 1], np.random.default_rng(0).integers(0, E, 7)]))
    wd = wt.double().numpy()
    rlp, rlse = LH.edge_logprob(h[rows].double().numpy(), wd, y[rows].numpy())
    assert np.abs(lse[rows].double().numpy() - rlse).max() <= TOL
    assert np.abs(lp[rows].double().numpy() - rlp).max() <= TOL
    assert bool((lp <= 1e-5).all()) and bool(torch.isfinite(lp).all())
    lp2, lse2, _ = _run(h, wt, y)
    assert torch.equal(lp2, lp) and torch.equal(lse2, lse)  # no atomics: identical on every run


def test_edge_logprob_bad_label_and_empty():
    x = W.draw_lm_head(4, 64, 300, seed=1)
    h, w, y = x["hidden_sel"], x["weight"], x["labels"].clone()
    y[2] = 300
    lp, lse, st = _run(h, w, y)
    assert st == spc.SP_DEV_INDEX_RANGE
    assert torch.isnan(lp[2]) and torch.isfinite(lp[[0, 1, 3]]).all()
    lp0, _, st0 = _run(h[:0], w, y[:0])
    assert st0 == 0 and lp0.numel() == 0


def test_edge_logprob_after_gather_on_tiny():
    """Gather the edge-source states, then project: the two kernels in sequence."""
    from oracle import gather as OG
    w = W.get("tiny")
    hid = W.draw_tensors(w, "bf16", with_hidden=True)["hidden"]
    idx = torch.from_numpy(w.edge_idx.astype(np.int32))
    sel = spc.edge_gather(hid.cuda(), idx.cuda())
    x = W.draw_lm_head(len(idx), w.hidden_dim, 1000, seed=5)
    lp, lse, st = _run(sel.cpu(), x["weight"], x["labels"])
    assert st == 0
    ref_sel = OG.edge_gather(hid.double().numpy(), w.edge_idx)
    rlp, _ = LH.edge_logprob(ref_sel, x["weight"].double().numpy(), x["labels"].numpy())
    assert np.abs(lp.double().numpy() - rlp).max() <= TOL


# ------------------------------------------------------------------ backward
#
# dlogits is rounded to bf16 (half an ulp: at most 2^-8 relative per element,
# about 2^-9 / sqrt(3) in rms for uniform rounding errors) before the two
# fp32-accumulated products, so d_hidden_sel and d_weight agree with the fp64
# oracle to a relative L2 error of about 1e-3; the tests use 5e-3 (the pages'
# gradient threshold is 2.5e-2).
GRAD_TOL = 5e-3


def _rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def _bwd(h, w, y, g):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    hc, wc, yc = h.cuda(), w.cuda(), y.cuda()
    _, lse = spc.edge_logprob(hc, wc, yc, st)
    dh, dw = spc.edge_logprob_bwd(hc, wc, yc, lse, g.cuda(), st)
    torch.cuda.synchronize()
    return dh.cpu(), dw.cpu(), st.item()


@pytest.mark.parametrize("E,V,Hd", [(1, 8, 8), (5, 304, 64), (300, 1000, 200), (129, 520, 136), (260, 4096, 512)])
def test_edge_logprob_bwd_matches_oracle(E, V, Hd):
    x = W.draw_lm_head(E, Hd, V, seed=E + 2 * V)
    h, w, y, g = x["hidden_sel"], x["weight"], x["labels"], x["grad_logprob"]
    dh, dw, st = _bwd(h, w, y, g)
    assert st == 0
    rdh, rdw = LH.edge_logprob_backward(h.double().numpy(), w.double().numpy(), y.numpy(), g.double().numpy())
    assert _rel_l2(dh, rdh) <= GRAD_TOL
    assert _rel_l2(dw, rdw) <= GRAD_TOL
    # vocabulary rows that no action samples get only the softmax part; the sampled ones the one-hot too
    for v in np.unique(y.numpy())[:3]:
        assert _rel_l2(dw[v], rdw[v]) <= 4 * GRAD_TOL


def test_edge_logprob_bwd_full_size_sampled_rows():
    """3419 actions, hidden 4096, vocabulary 131,072: all lse, sampled d_hidden_sel and d_weight rows."""
    w = W.get("agent")
    E = len(w.edge_idx)
    x = W.draw_lm_head(E, w.hidden_dim, seed=4)
    h, wt, y, g = x["hidden_sel"], x["weight"], x["labels"], x["grad_logprob"]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    hc, wc, yc = h.cuda(), wt.cuda(), y.cuda()
    lp, lse = spc.edge_logprob(hc, wc, yc, st)
    dh, dw = spc.edge_logprob_bwd(hc, wc, yc, lse, g.cuda(), st)
    torch.cuda.synchronize()
    assert st.item() == 0
    hd, wd, yn, gd = h.double().numpy(), wt.double().numpy(), y.numpy(), g.double().numpy()
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 127, 128, E - 1], rng.integers(0, E, 6)]))
    rdh, _ = LH.edge_logprob_backward(hd[rows], wd, yn[rows], gd[rows])  # rows of d_hidden_sel are independent
    assert _rel_l2(dh.cpu()[rows], rdh) <= GRAD_TOL
    vrows = np.unique(np.concatenate([yn[:4], [0, 255, 256, 131071], rng.integers(0, 131072, 4)]))
    rdw = LH.weight_grad_rows(hd, wd, yn, gd, vrows)
    assert _rel_l2(dw.cpu()[vrows], rdw) <= GRAD_TOL
    assert torch.isfinite(dw).all() and torch.isfinite(dh).all()


def test_edge_logprob_bwd_skips_outputs_and_handles_no_actions():
    x = W.draw_lm_head(6, 64, 296, seed=2)
    h, w, y, g = (x[k].cuda() for k in ("hidden_sel", "weight", "labels", "grad_logprob"))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, lse = spc.edge_logprob(h, w, y, st)
    ws = torch.empty(spc.sp_edge_logprob_bwd_workspace_bytes(6, 296), dtype=torch.uint8, device="cuda")
    dh = torch.full((6, 64), 7.0, device="cuda")
    spc.sp_edge_logprob_bwd(h, w, y, lse, g, dh, None, ws, st)
    dh_all, _ = spc.edge_logprob_bwd(h, w, y, lse, g, st)
    torch.cuda.synchronize()
    assert torch.equal(dh, dh_all) and st.item() == 0
    dw0 = torch.full((296, 64), 7.0, device="cuda")
    spc.sp_edge_logprob_bwd(h[:0], w, y[:0], lse[:0], g[:0], None, dw0, ws, st)
    torch.cuda.synchronize()
    assert (dw0 == 0).all()
