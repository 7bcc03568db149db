"""The Python binding's marshalling, checked on the CPU.

Fake CUDA tensors carry a shape, dtype, device and data pointer.  The C entry
points are replaced by recorders and torch's device guard and current stream
by fakes.  Each binding call must then pass the tensors' pointers, sizes and
the stream of the tensors' own device, in the header's argument order, with
that device current.  Nothing reaches the library or a GPU.
"""
import contextlib
import math

import pytest
import torch

spc = pytest.importorskip("shared_prefix_causal_gb300")


class FakeCuda:
    is_cuda = True

    def __init__(self, shape, dtype, ptr, device=1):
        self.shape = tuple(shape)
        self.dtype = dtype
        self.ptr = ptr
        self.device = torch.device("cuda", device)

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return self.ptr

    def numel(self):
        return math.prod(self.shape)

    def element_size(self):
        return torch.empty(0, dtype=self.dtype).element_size()


@pytest.fixture
def fake_cuda(monkeypatch):
    entered = []

    @contextlib.contextmanager
    def device(d):
        entered.append(torch.device(d))
        yield

    class Stream:
        def __init__(self, d):
            self.cuda_stream = 0x5000 + (torch.device(d).index if d is not None else 0)

    monkeypatch.setattr(torch.cuda, "device", device)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda d=None: Stream(d))
    return entered


def _record(monkeypatch, name):
    calls = []

    def fn(*args):
        calls.append([a.value if hasattr(a, "value") else a for a in args])
        return 0

    monkeypatch.setattr(spc, name, fn)
    return calls


class FakePlan:
    handle = 0x77


def _attn_tensors(T=40, Hq=8, Hkv=2, D=64, dtype=torch.bfloat16):
    q = FakeCuda((T, Hq, D), dtype, 0x1000)
    k = FakeCuda((T, Hkv, D), dtype, 0x2000)
    v = FakeCuda((T, Hkv, D), dtype, 0x3000)
    o = FakeCuda((T, Hq, D), dtype, 0x4000)
    lse = FakeCuda((Hq, T), torch.float32, 0x5000)
    return q, k, v, o, lse


def test_forward_marshalling(monkeypatch, fake_cuda):
    calls = _record(monkeypatch, "_c_fwd")
    q, k, v, o, lse = _attn_tensors()
    st = FakeCuda((1,), torch.int32, 0x9000)
    spc.sp_tree_attn_fwd(FakePlan(), q, k, v, o, lse, 0.125, st)
    (c,) = calls
    assert c[:7] == [0x77, spc.SP_BF16, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000]
    assert c[7:11] == [40, 8, 2, 64] and c[11] == pytest.approx(0.125)
    assert c[12:] == [0x9000, 0x5001]  # d_status; the current stream of the tensors' device (cuda:1)
    assert fake_cuda == [torch.device("cuda", 1)]


@pytest.mark.parametrize("variant", ["atomic", "deterministic"])
def test_backward_marshalling(monkeypatch, fake_cuda, variant):
    calls = _record(monkeypatch, "_c_bwd" if variant == "atomic" else "_c_bwd_det")
    q, k, v, o, lse = _attn_tensors(dtype=torch.float32)
    do = FakeCuda(q.shape, q.dtype, 0x6000)
    dq, dk, dv = FakeCuda(q.shape, q.dtype, 0x7000), FakeCuda(k.shape, k.dtype, 0x7100), FakeCuda(v.shape, v.dtype, 0x7200)
    ws = FakeCuda((4096,), torch.uint8, 0x8000)
    fn = spc.sp_tree_attn_bwd if variant == "atomic" else spc.sp_tree_attn_bwd_deterministic
    fn(FakePlan(), q, k, v, o, lse, do, dq, dk, dv, ws, 0.5, None, 0x1234)
    (c,) = calls
    assert c[:13] == [0x77, spc.SP_F32, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x7100, 0x7200,
                      0x8000, 4096]
    assert c[13:17] == [40, 8, 2, 64] and c[17] == pytest.approx(0.5)
    assert c[18:] == [None, 0x1234]  # no status word; the explicit stream handle
    assert fake_cuda == [torch.device("cuda", 1)]


def test_noalloc_backward_marshalling(monkeypatch, fake_cuda):
    calls = _record(monkeypatch, "_c_bwd_noalloc")
    q, k, v, o, lse = _attn_tensors()
    do = FakeCuda(q.shape, q.dtype, 0x6000)
    dq, dk, dv = FakeCuda(q.shape, q.dtype, 0x7000), FakeCuda(k.shape, k.dtype, 0x7100), FakeCuda(v.shape, v.dtype, 0x7200)
    spc.sp_tree_attn_bwd_noalloc(FakePlan(), q, k, v, o, lse, do, dq, dk, dv, 0.25)
    (c,) = calls
    assert c[:11] == [0x77, spc.SP_BF16, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x7100, 0x7200]
    assert c[11:15] == [40, 8, 2, 64] and c[16:] == [None, 0x5001]


def test_gather_marshalling(monkeypatch, fake_cuda):
    calls = _record(monkeypatch, "_c_gather")
    hidden = FakeCuda((100, 256), torch.bfloat16, 0x1000, device=0)
    idx = FakeCuda((7,), torch.int32, 0x2000, device=0)
    out = FakeCuda((7, 256), torch.bfloat16, 0x3000, device=0)
    spc.sp_edge_gather(hidden, idx, out)
    assert calls == [[spc.SP_BF16, 0x1000, 100, 256, 0x2000, 7, 0x3000, None, 0x5000]]
    assert fake_cuda == [torch.device("cuda", 0)]


def test_gather_backward_marshalling(monkeypatch, fake_cuda):
    calls = _record(monkeypatch, "_c_gather_bwd")
    g = FakeCuda((7, 256), torch.bfloat16, 0x1000)
    idx = FakeCuda((7,), torch.int32, 0x2000)
    gh = FakeCuda((100, 256), torch.bfloat16, 0x3000)
    ws = FakeCuda((1024,), torch.uint8, 0x4000)
    spc.sp_edge_gather_bwd(g, idx, gh, ws)
    assert calls == [[spc.SP_BF16, 0x1000, 7, 256, 0x2000, 100, 0x3000, 0x4000, 1024, None, 0x5001]]


def test_vocabulary_head_marshalling(monkeypatch, fake_cuda):
    fwd = _record(monkeypatch, "_c_lmh")
    bwd = _record(monkeypatch, "_c_lmh_bwd")
    h = FakeCuda((5, 64), torch.bfloat16, 0x1000)
    w = FakeCuda((96, 64), torch.bfloat16, 0x2000)
    y = FakeCuda((5,), torch.int32, 0x3000)
    lp, lse, g = (FakeCuda((5,), torch.float32, p) for p in (0x4000, 0x5000, 0x6000))
    ws = FakeCuda((2048,), torch.uint8, 0x7000)
    dh, dw = FakeCuda((5, 64), torch.float32, 0x8000), FakeCuda((96, 64), torch.float32, 0x9000)
    spc.sp_edge_logprob(h, w, y, lp, lse, ws)
    spc.sp_edge_logprob_bwd(h, w, y, lse, g, dh, dw, ws)
    assert fwd == [[spc.SP_BF16, 0x1000, 5, 64, 0x2000, 96, 0x3000, 0x4000, 0x5000, 0x7000, 2048, None, 0x5001]]
    assert bwd == [[spc.SP_BF16, 0x1000, 5, 64, 0x2000, 96, 0x3000, 0x5000, 0x6000, 0x8000, 0x9000, 0x7000, 2048,
                    None, 0x5001]]
    assert fake_cuda == [torch.device("cuda", 1)] * 2


def test_plan_upload_to_marshalling(monkeypatch, fake_cuda):
    calls = _record(monkeypatch, "_c_plan_upload_to")
    buf = FakeCuda((1 << 16,), torch.uint8, 0xA000)
    spc.sp_plan_upload_to(FakePlan(), buf)
    assert calls == [[0x77, 0xA000, 1 << 16, 0x5001]]
    assert fake_cuda == [torch.device("cuda", 1)]


def test_shape_and_dtype_mismatches_raise_before_the_call(monkeypatch, fake_cuda):
    calls = _record(monkeypatch, "_c_fwd")
    q, k, v, o, lse = _attn_tensors()
    bad_o = FakeCuda(o.shape, torch.float32, o.ptr)
    bad_lse = FakeCuda((lse.shape[1], lse.shape[0]), torch.float32, lse.ptr)
    for args in ((q, k, v, bad_o, lse), (q, k, v, o, bad_lse)):
        with pytest.raises(ValueError):
            spc.sp_tree_attn_fwd(FakePlan(), *args, 0.1)
    with pytest.raises(ValueError):
        spc.sp_tree_attn_fwd(FakePlan(), torch.zeros(4, 8, 64), k, v, o, lse, 0.1)  # a CPU tensor
    assert calls == [] and fake_cuda == []


@pytest.mark.parametrize("entry", ["sp_tree_attn_bwd", "sp_tree_attn_bwd_deterministic", "sp_tree_attn_bwd_noalloc"])
def test_backward_refuses_a_bad_lse_or_status_word(monkeypatch, fake_cuda, entry):
    """An lse of the wrong dtype or size would be read past its end by the kernels; a status word
    that is not int32 would be written with the wrong width.  Both are refused before the C call."""
    recorders = [_record(monkeypatch, n) for n in ("_c_bwd", "_c_bwd_det", "_c_bwd_noalloc")]
    q, k, v, o, lse = _attn_tensors()
    do = FakeCuda(q.shape, q.dtype, 0x6000)
    dq, dk, dv = FakeCuda(q.shape, q.dtype, 0x7000), FakeCuda(k.shape, k.dtype, 0x7100), FakeCuda(v.shape, v.dtype, 0x7200)
    ws = FakeCuda((4096,), torch.uint8, 0x8000)
    fn = getattr(spc, entry)

    def call(lse_, st=None):
        if entry == "sp_tree_attn_bwd_noalloc":
            fn(FakePlan(), q, k, v, o, lse_, do, dq, dk, dv, 0.25, st)
        else:
            fn(FakePlan(), q, k, v, o, lse_, do, dq, dk, dv, ws, 0.25, st)

    bad = [FakeCuda(lse.shape, torch.bfloat16, lse.ptr),                  # wrong dtype
           FakeCuda((lse.shape[0], lse.shape[1] - 1), torch.float32, lse.ptr),  # one token short
           FakeCuda((lse.shape[1], lse.shape[0]), torch.float32, lse.ptr)]      # transposed
    for b in bad:
        with pytest.raises(ValueError):
            call(b)
    with pytest.raises(ValueError):
        call(lse, FakeCuda((1,), torch.int64, 0x9000))
    assert all(r == [] for r in recorders) and fake_cuda == []
    call(lse, FakeCuda((1,), torch.int32, 0x9000))  # the good case reaches the library
    assert sum(len(r) for r in recorders) == 1
