"""The allocation-free backward entry point (sp_tree_attn_bwd_noalloc).

Some callers cannot allocate device memory (a memory pool that owns the whole
device, a runtime with a fixed footprint, a plugin handed only its buffers),
so they cannot hand sp_tree_attn_bwd a workspace; this entry point uses the
library's own fixed device scratch instead.  Checked here, through the C ABI:

* its dK and dV equal the workspace entry point's bit for bit (the same
  kernels; dK and dV are formed per key block without atomics), and its dQ
  (fp32 atomics, so the order of additions varies) is within 5e-3 relative L2
  of it; in fp32 every output is bit-equal;
* it matches the fp64 oracle within the parity bounds;
* a second call after a call of another size, which leaves other contents in
  the shared scratch, gives the same results as the first;
* the second call on a device commits no device memory (free bytes unchanged);
* sizes whose scratch need exceeds the fixed size are refused.

Collected last on purpose, so that a run stopping at its first failure has
run every other test before this one.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A

pytestmark = pytest.mark.gpu

spc = pytest.importorskip("shared_prefix_causal_gb300")

ORACLE_TOL = {"bf16": 2.5e-2, "f32": 1e-5}  # the relative-L2 bounds of the parity tests
DQ_TOL = 5e-3  # dQ against the workspace entry point (same kernels, atomics in another order)


def _rel(a, b):
    a = a.double().cpu()
    b = b.double().cpu()
    return float((a - b).norm() / b.norm())


def _setup(w, dtype):
    x = W.draw_tensors(w, dtype)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    G = w.hq // w.hkv
    plan = spc.tree_plan(w.tree, 128 // G, 128, 0)
    o, lse = spc.tree_attn_fwd(plan, q, k, v, w.softmax_scale)
    return x, plan, (q, k, v, o, lse, do)


def _noalloc(w, plan, t, outs, st):
    q, k, v, o, lse, do = t
    spc.sp_tree_attn_bwd_noalloc(plan, q, k, v, o, lse, do, *outs, w.softmax_scale, st)


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


def _gqa_workload():
    rng = np.random.default_rng(21)
    tree = W.random_small_tree(rng, max_segments=24, max_len=300)
    return W.Workload("noalloc", "", tree, 8, 2, 128, 0.5, 21, None, None)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_tiny_repeated_calls_with_another_size_between(dtype):
    w = W.tiny()
    x, plan, t = _setup(w, dtype)
    q, k, v, o, lse, do = t
    ref = spc.tree_attn_bwd(plan, q, k, v, o, lse, do, w.softmax_scale)  # workspace entry point
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    first = tuple(torch.empty_like(a) for a in (q, k, v))
    second = tuple(torch.empty_like(a) for a in (q, k, v))
    # a call of another size in between leaves other contents in the shared scratch
    w2 = _gqa_workload()
    _, plan2, t2 = _setup(w2, "bf16")
    outs2 = tuple(torch.empty_like(a) for a in (t2[0], t2[1], t2[2]))

    _noalloc(w, plan, t, first, st)
    _noalloc(w2, plan2, t2, outs2, st)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    _noalloc(w, plan, t, second, st)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert st.item() == 0
    assert free_after == free_before, "the second call committed device memory"

    for got in (first, second):
        dq, dk, dv = got
        assert _same_bits(dk, ref[1]) and _same_bits(dv, ref[2])
        if dtype == "f32":
            assert _same_bits(dq, ref[0])
        else:
            assert _rel(dq, ref[0]) <= DQ_TOL

    # and against the fp64 oracle directly
    tr = w.tree
    xs = {n: x[n].float().numpy() for n in ("q", "k", "v", "do")}
    want = A.tree_backward(xs["q"], xs["k"], xs["v"], xs["do"], tr.seg_start, tr.seg_len, tr.parent,
                           w.softmax_scale)
    for got, ref64 in zip(second, want):
        err = float(np.linalg.norm(got.double().cpu().numpy() - ref64) / np.linalg.norm(ref64))
        assert err <= ORACLE_TOL[dtype]


def test_noalloc_matches_workspace_entry_point_gqa_tree():
    w = _gqa_workload()
    assert spc.sp_tree_attn_bwd_workspace_bytes(spc.SP_BF16, w.T, w.hq, 128) <= spc.NOALLOC_SCRATCH_BYTES
    _, plan, t = _setup(w, "bf16")
    q, k, v, o, lse, do = t
    ref = spc.tree_attn_bwd(plan, q, k, v, o, lse, do, w.softmax_scale)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        got = tuple(torch.empty_like(a) for a in (q, k, v))
        _noalloc(w, plan, t, got, st)
        torch.cuda.synchronize()
        assert st.item() == 0
        assert _same_bits(got[1], ref[1]) and _same_bits(got[2], ref[2])
        assert _rel(got[0], ref[0]) <= DQ_TOL


def test_noalloc_rejects_sizes_beyond_its_scratch():
    T, Hq, Hkv, D = 200000, 32, 8, 128  # 4 * T * Hq * (D + 1) bytes > 64 MiB
    assert spc.sp_tree_attn_bwd_workspace_bytes(spc.SP_BF16, T, Hq, D) > spc.NOALLOC_SCRATCH_BYTES
    tree = W.tree_from_preorder([T], [-1])
    plan = spc.tree_plan(tree, 128 // 4, 128, 0, upload=False)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check fails first
    rc = spc._c_bwd_noalloc(plan.handle, spc.SP_BF16, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                            T, Hq, Hkv, D, 0.088, None, None)
    assert rc == -8  # SP_ERR_WORKSPACE
