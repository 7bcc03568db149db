"""Failure detection without a GPU fault.

Host side: malformed input is rejected before any launch (see test_abi.py for
the tree and argument checks).  Device side: every wait in the tensor-core
kernels is bounded; a wait that can never complete must come back as
SP_DEV_TIMEOUT in the status word, and the context must stay usable."""
import pytest
import torch

import workloads as W

spc = pytest.importorskip("shared_prefix_causal_gb300")


def test_wait_timeout_rejects_bad_arguments():
    assert spc._c_wait_timeout(10, None, None) == -2  # checked before any launch


@pytest.mark.gpu
def test_bounded_wait_reports_timeout_and_context_survives():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    spc.sp_debug_wait_timeout(1 << 12, st)
    torch.cuda.synchronize()
    assert st.item() == spc.SP_DEV_TIMEOUT
    # the same context still runs attention correctly afterwards
    w = W.tiny()
    x = W.draw_tensors(w, "bf16")
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    plan = spc.tree_plan(w.tree, 128 // (w.hq // w.hkv), 128, 0)
    st.zero_()
    o, lse = spc.tree_attn_fwd(plan, q, k, v, w.softmax_scale, st)
    torch.cuda.synchronize()
    assert st.item() == 0 and torch.isfinite(o.float()).all()
