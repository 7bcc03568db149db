"""The allocation-free backward entry point (sp_tree_attn_bwd_noalloc).

Some callers cannot allocate device memory, so cannot hand sp_tree_attn_bwd
a workspace; this entry point uses the library's own fixed device scratch
instead.  It must give the same results as the workspace entry point, on
repeated calls (the scratch keeps the previous call's contents), and refuse
sizes whose scratch need exceeds the fixed size.  Collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

spc = pytest.importorskip("shared_prefix_causal_gb300")

TOL = {"bf16": 2.5e-2, "f32": 1e-5}  # the relative-L2 bounds of the parity tests


def _rel(a, b):
    a = a.double().cpu()
    b = b.double().cpu()
    return float((a - b).norm() / b.norm())


def _case(w, dtype):
    x = W.draw_tensors(w, dtype)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    G = w.hq // w.hkv
    plan = spc.tree_plan(w.tree, 128 // G, 128, 0)
    o, lse = spc.tree_attn_fwd(plan, q, k, v, w.softmax_scale)
    ref = spc.tree_attn_bwd(plan, q, k, v, o, lse, do, w.softmax_scale)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        spc.sp_tree_attn_bwd_noalloc(plan, q, k, v, o, lse, do, dq, dk, dv, w.softmax_scale, st)
        outs.append((dq, dk, dv))
    torch.cuda.synchronize()
    assert st.item() == 0
    for got in outs:
        for a, b in zip(got, ref):
            assert _rel(a, b) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_workspace_entry_point_tiny(dtype):
    _case(W.tiny(), dtype)


def test_noalloc_matches_workspace_entry_point_gqa_tree():
    rng = np.random.default_rng(21)
    tree = W.random_small_tree(rng, max_segments=24, max_len=300)
    w = W.Workload("noalloc", "", tree, 8, 2, 128, 0.5, 21, None, None)
    assert spc.sp_tree_attn_bwd_workspace_bytes(spc.SP_BF16, w.T, w.hq, 128) <= spc.NOALLOC_SCRATCH_BYTES
    _case(w, "bf16")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    T, Hq, Hkv, D = 200000, 32, 8, 128  # 4 * T * Hq * (D + 1) bytes > 64 MiB
    assert spc.sp_tree_attn_bwd_workspace_bytes(spc.SP_BF16, T, Hq, D) > spc.NOALLOC_SCRATCH_BYTES
    tree = W.tree_from_preorder([T], [-1])
    plan = spc.tree_plan(tree, 128 // 4, 128, 0, upload=False)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check fails first
    rc = spc._c_bwd_noalloc(plan.handle, spc.SP_BF16, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                            T, Hq, Hkv, D, 0.088, None, None)
    assert rc == -8  # SP_ERR_WORKSPACE
