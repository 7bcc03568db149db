"""Python binding of the shared-prefix tree attention C ABI (``libspc.so``).

Argument marshalling only: every function here checks Python-side types,
pulls raw pointers, sizes and the current CUDA stream out of torch tensors and
calls the C entry point of the same name (declared in
``include/shared_prefix_causal.h``).  All arithmetic runs in the library's
CUDA kernels.  There is no fallback: if ``libspc.so`` is missing, importing
this package raises.  Build it with ``python shared_prefix_causal_gb300/build.py``.

Layouts: q, o, dO, dq ``[T, Hq, D]``; k, v, dk, dv ``[T, Hkv, D]``; lse
``[Hq, T]`` fp32; hidden ``[T, hidden_dim]``; edge indices int32 ``[E]``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspc.so")

SP_OK = 0
SP_BF16 = 0
SP_F32 = 1
SP_DEV_INDEX_RANGE = 1
SP_DEV_TIMEOUT = 2
SP_DEV_BAD_PLAN = 4
SP_DEV_SMEM_LAYOUT = 8
SP_ERR_CAP = -10

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run `python shared_prefix_causal_gb300/build.py` "
                      "(the CUDA library is required: there is no CPU path)")

_lib = ctypes.CDLL(LIB_PATH)
_i32 = ctypes.c_int32
_vp = ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int32)


class _TreeDesc(ctypes.Structure):
    _fields_ = [("num_segments", _i32), ("total_tokens", _i32), ("seg_start", _i32p),
                ("seg_len", _i32p), ("parent", _i32p), ("depth", _i32p)]


class _PlanInfo(ctypes.Structure):
    _fields_ = [("tile_tokens", _i32), ("kv_block", _i32), ("order", _i32), ("total_tokens", _i32),
                ("num_segments", _i32), ("n_tiles", _i32), ("n_ranges", _i32), ("n_bwd", _i32),
                ("max_ranges_per_tile", _i32), ("tiles", _i32p), ("ranges", _i32p), ("bwd", _i32p)]


class _FragInfo(ctypes.Structure):
    _fields_ = [("num_fragments", _i32), ("num_entries", _i32), ("physical_tokens", ctypes.c_int64),
                ("fragment_tokens", ctypes.c_int64), ("offsets", _i32p), ("tokens", _i32p), ("seg", _i32p),
                ("owned", _i32p), ("local_parent", _i32p), ("local_start", _i32p)]


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


_c_tree_plan = _sig("sp_tree_plan", ctypes.c_int, [ctypes.POINTER(_TreeDesc), _i32, _i32, _i32, ctypes.POINTER(_vp)])
_c_plan_view = _sig("sp_plan_view", ctypes.c_int, [_vp, ctypes.POINTER(_PlanInfo)])
_c_plan_upload = _sig("sp_plan_upload", ctypes.c_int, [_vp, _vp])
_c_plan_destroy = _sig("sp_plan_destroy", None, [_vp])
_c_fwd = _sig("sp_tree_attn_fwd", ctypes.c_int,
              [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, ctypes.c_float, _vp, _vp])
_c_fwd_paired = _sig("sp_tree_attn_fwd_paired", ctypes.c_int,
                     [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, ctypes.c_float, _vp, _vp])
_c_ws = _sig("sp_tree_attn_bwd_workspace_bytes", ctypes.c_size_t, [_i32, _i32, _i32, _i32])
_c_bwd = _sig("sp_tree_attn_bwd", ctypes.c_int,
              [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
               _i32, _i32, _i32, _i32, ctypes.c_float, _vp, _vp])
_c_plan_bytes = _sig("sp_plan_device_bytes", ctypes.c_size_t, [_vp])
_c_plan_bwd_blocks = _sig("sp_plan_bwd_blocks", ctypes.c_int,
                          [_vp, ctypes.POINTER(ctypes.POINTER(ctypes.c_int32)), ctypes.POINTER(ctypes.c_int32),
                           ctypes.POINTER(ctypes.POINTER(ctypes.c_int32))])
_c_plan_upload_to = _sig("sp_plan_upload_to", ctypes.c_int, [_vp, _vp, ctypes.c_size_t, _vp])
_c_frag_plan = _sig("sp_fragment_plan", ctypes.c_int,
                    [ctypes.POINTER(_TreeDesc), ctypes.c_int64, ctypes.POINTER(ctypes.c_void_p)])
_c_frag_view = _sig("sp_fragment_view", ctypes.c_int, [_vp, ctypes.POINTER(_FragInfo)])
_c_frag_destroy = _sig("sp_fragment_destroy", None, [_vp])
_c_bwd_det = _sig("sp_tree_attn_bwd_deterministic", ctypes.c_int,
                  [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                   _i32, _i32, _i32, _i32, ctypes.c_float, _vp, _vp])
_c_bwd_timed = _sig("sp_tree_attn_bwd_timed", ctypes.c_int,
                    [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                     _i32, _i32, _i32, _i32, ctypes.c_float, _i32, _vp, _vp, _vp, _vp])
_c_bwd_noalloc = _sig("sp_tree_attn_bwd_noalloc", ctypes.c_int,
                      [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                       _i32, _i32, _i32, _i32, ctypes.c_float, _vp, _vp])
_c_gather = _sig("sp_edge_gather", ctypes.c_int, [_i32, _vp, _i32, _i32, _vp, _i32, _vp, _vp, _vp])
_c_status = _sig("sp_status_string", ctypes.c_char_p, [ctypes.c_int])
_c_lmh_ws = _sig("sp_edge_logprob_workspace_bytes", ctypes.c_size_t, [_i32, _i32])
_c_lmh = _sig("sp_edge_logprob", ctypes.c_int,
              [_i32, _vp, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp])
_c_lmh_bwd_ws = _sig("sp_edge_logprob_bwd_workspace_bytes", ctypes.c_size_t, [_i32, _i32])
_c_lmh_bwd = _sig("sp_edge_logprob_bwd", ctypes.c_int,
                  [_i32, _vp, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp])
_c_gather_bwd_ws = _sig("sp_edge_gather_bwd_workspace_bytes", ctypes.c_size_t, [_i32, _i32])
_c_gather_bwd = _sig("sp_edge_gather_bwd", ctypes.c_int,
                     [_i32, _vp, _i32, _i32, _vp, _i32, _vp, _vp, ctypes.c_size_t, _vp, _vp])
_c_wait_timeout = _sig("sp_debug_wait_timeout", ctypes.c_int, [_i32, _vp, _vp])
_c_cta_clock = _sig("sp_debug_cta_clock", ctypes.c_int, [_i32, _vp, ctypes.c_int64])

EXPORTED = ("sp_tree_plan", "sp_plan_view", "sp_plan_upload", "sp_plan_destroy", "sp_tree_attn_fwd",
            "sp_tree_attn_bwd_workspace_bytes", "sp_tree_attn_bwd", "sp_tree_attn_bwd_noalloc", "sp_edge_gather",
            "sp_status_string", "sp_debug_wait_timeout", "sp_edge_gather_bwd_workspace_bytes", "sp_edge_gather_bwd",
            "sp_edge_logprob_workspace_bytes", "sp_edge_logprob", "sp_edge_logprob_bwd_workspace_bytes",
            "sp_edge_logprob_bwd", "sp_tree_attn_bwd_deterministic", "sp_fragment_plan", "sp_fragment_view",
            "sp_fragment_destroy", "sp_plan_device_bytes", "sp_plan_upload_to", "sp_tree_attn_bwd_timed",
            "sp_debug_cta_clock", "sp_tree_attn_fwd_paired", "sp_plan_bwd_blocks")
NOALLOC_SCRATCH_BYTES = 64 << 20


class SPError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {sp_status_string(code)} (status {code})")
        self.code = code


def sp_status_string(code: int) -> str:
    return _c_status(int(code)).decode()


def _check(code: int, where: str):
    if code != SP_OK:
        raise SPError(code, where)


class Plan:
    """Owner of an ``sp_plan`` handle (freed with ``sp_plan_destroy``)."""

    def __init__(self, handle: int):
        self._h = _vp(handle)

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            _c_plan_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def info(self) -> dict:
        return sp_plan_view(self)


def sp_tree_plan(seg_start, seg_len, parent, depth, tile_tokens: int, kv_block: int, order: int = 0) -> Plan:
    arrs = [np.ascontiguousarray(np.asarray(a, dtype=np.int32)) for a in (seg_start, seg_len, parent, depth)]
    n = int(arrs[0].shape[0])
    total = int(arrs[1].astype(np.int64).sum()) if n else 0
    ptr = [a.ctypes.data_as(_i32p) for a in arrs]
    desc = _TreeDesc(n, total, *ptr)
    out = _vp()
    _check(_c_tree_plan(ctypes.byref(desc), tile_tokens, kv_block, order, ctypes.byref(out)), "sp_tree_plan")
    return Plan(out.value)


def sp_plan_view(plan: Plan) -> dict:
    info = _PlanInfo()
    _check(_c_plan_view(plan.handle, ctypes.byref(info)), "sp_plan_view")

    def arr(p, n, w):
        if n == 0:
            return np.zeros((0, w), dtype=np.int32)
        return np.ctypeslib.as_array(p, shape=(n * w,)).reshape(n, w).copy()

    return {
        "tile_tokens": info.tile_tokens, "kv_block": info.kv_block, "order": info.order,
        "total_tokens": info.total_tokens, "num_segments": info.num_segments,
        "max_ranges_per_tile": info.max_ranges_per_tile,
        "tiles": arr(info.tiles, info.n_tiles, 5), "ranges": arr(info.ranges, info.n_ranges, 2),
        "bwd": arr(info.bwd, info.n_bwd, 5),
    }


def sp_plan_bwd_blocks(plan: Plan) -> dict:
    """The key blocks the bf16 backward runs ([n][5], launch order) and every key's query-run end."""
    rows, keys = ctypes.POINTER(ctypes.c_int32)(), ctypes.POINTER(ctypes.c_int32)()
    n = ctypes.c_int32()
    _check(_c_plan_bwd_blocks(plan.handle, ctypes.byref(rows), ctypes.byref(n), ctypes.byref(keys)),
           "sp_plan_bwd_blocks")
    T = int(sp_plan_view(plan)["total_tokens"])
    return {
        "rows": np.ctypeslib.as_array(rows, shape=(n.value * 5,)).reshape(n.value, 5).copy()
        if n.value else np.zeros((0, 5), dtype=np.int32),
        "key_end": np.ctypeslib.as_array(keys, shape=(T,)).copy() if T else np.zeros(0, dtype=np.int32),
    }


def _stream(stream, device=None):
    """The stream argument as a cudaStream_t: None means the current stream of ``device``."""
    import torch
    if stream is None:
        return _vp(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, int):
        return _vp(stream)
    return _vp(stream.cuda_stream)


def _on(t):
    """Makes tensor t's GPU current for one call: the library launches on the current device."""
    import torch
    return torch.cuda.device(t.device)


def sp_plan_upload(plan: Plan, stream=None):
    _check(_c_plan_upload(plan.handle, _stream(stream)), "sp_plan_upload")


def sp_plan_device_bytes(plan: Plan) -> int:
    return int(_c_plan_bytes(plan.handle))


def sp_plan_upload_to(plan: Plan, buffer, stream=None):
    """Upload the plan into a caller-owned device buffer (a CUDA uint8 tensor kept alive by the caller)."""
    _need_cuda(buffer)
    with _on(buffer):
        _check(_c_plan_upload_to(plan.handle, _ptr(buffer), buffer.numel() * buffer.element_size(),
                                 _stream(stream, buffer.device)), "sp_plan_upload_to")


def _ptr(t):
    return _vp(t.data_ptr()) if t is not None else _vp()


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return SP_BF16
    if t.dtype == torch.float32:
        return SP_F32
    return -1


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _need_status(d_status):
    """The optional device status word: one int32 (the kernels OR their error bits into it)."""
    import torch
    if d_status is not None and (d_status.dtype != torch.int32 or d_status.numel() < 1):
        raise ValueError("d_status must be an int32 CUDA tensor of at least one element")


def _check_bwd_shapes(q, k, v, o, lse, d_o, dq, dk, dv):
    """Shapes and dtypes the backward entry points read and write: (T, Hq, Hkv, D)."""
    import torch
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    for t, shp in ((k, (T, Hkv, D)), (v, (T, Hkv, D)), (o, (T, Hq, D)), (d_o, (T, Hq, D)), (dq, (T, Hq, D)),
                   (dk, (T, Hkv, D)), (dv, (T, Hkv, D))):
        if tuple(t.shape) != shp or t.dtype != q.dtype:
            raise ValueError("shape or dtype mismatch")
    if tuple(lse.shape) != (Hq, T) or lse.dtype != torch.float32:
        raise ValueError("lse must be float32 [Hq, T]")
    return T, Hq, Hkv, D


def sp_tree_attn_fwd(plan: Plan, q, k, v, o, lse, softmax_scale: float, d_status=None, stream=None, _fn=None):
    import torch
    _need_cuda(q, k, v, o, lse, d_status)
    _need_status(d_status)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (T, Hkv, D) or tuple(v.shape) != (T, Hkv, D) or tuple(o.shape) != (T, Hq, D) \
            or tuple(lse.shape) != (Hq, T) or o.dtype != q.dtype or k.dtype != q.dtype or v.dtype != q.dtype \
            or lse.dtype != torch.float32:
        raise ValueError("shape or dtype mismatch")
    fn, name = _fn or (_c_fwd, "sp_tree_attn_fwd")
    with _on(q):
        _check(fn(plan.handle, _dtype_code(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), T, Hq, Hkv, D,
                  float(softmax_scale), _ptr(d_status), _stream(stream, q.device)), name)


def sp_tree_attn_fwd_paired(plan: Plan, q, k, v, o, lse, softmax_scale: float, d_status=None, stream=None):
    """sp_tree_attn_fwd on pairs of SMs (cta_group::2 products); bf16, head_dim 128."""
    sp_tree_attn_fwd(plan, q, k, v, o, lse, softmax_scale, d_status, stream,
                     _fn=(_c_fwd_paired, "sp_tree_attn_fwd_paired"))


def sp_tree_attn_bwd_workspace_bytes(dtype: int, T: int, Hq: int, D: int) -> int:
    return int(_c_ws(dtype, T, Hq, D))


def sp_tree_attn_bwd(plan: Plan, q, k, v, o, lse, d_o, dq, dk, dv, workspace, softmax_scale: float,
                     d_status=None, stream=None, _fn=None):
    _need_cuda(q, k, v, o, lse, d_o, dq, dk, dv, workspace, d_status)
    _need_status(d_status)
    T, Hq, Hkv, D = _check_bwd_shapes(q, k, v, o, lse, d_o, dq, dk, dv)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    fn, name = _fn or (_c_bwd, "sp_tree_attn_bwd")
    with _on(q):
        _check(fn(plan.handle, _dtype_code(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o),
                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), ws_bytes, T, Hq, Hkv, D, float(softmax_scale),
                  _ptr(d_status), _stream(stream, q.device)), name)


def sp_tree_attn_bwd_deterministic(plan: Plan, q, k, v, o, lse, d_o, dq, dk, dv, workspace, softmax_scale: float,
                                   d_status=None, stream=None):
    """sp_tree_attn_bwd with dQ formed per query tile (no atomics): identical bits on every run."""
    sp_tree_attn_bwd(plan, q, k, v, o, lse, d_o, dq, dk, dv, workspace, softmax_scale, d_status, stream,
                     _fn=(_c_bwd_det, "sp_tree_attn_bwd_deterministic"))


def sp_tree_attn_bwd_timed(plan: Plan, q, k, v, o, lse, d_o, dq, dk, dv, workspace, softmax_scale: float,
                           deterministic: bool, ev_main_begin, ev_main_end, d_status=None, stream=None):
    """sp_tree_attn_bwd(_deterministic) with two caller-owned events recorded around its main kernel.

    The events are ``torch.cuda.Event(enable_timing=True)`` objects or raw ``cudaEvent_t`` handles (ints).
    torch creates an event's handle at its first record, so a torch event never recorded before is recorded
    once on the current stream here; the library then records it again around the main kernel."""
    _need_cuda(q, k, v, o, lse, d_o, dq, dk, dv, workspace, d_status)
    _need_status(d_status)
    T, Hq, Hkv, D = _check_bwd_shapes(q, k, v, o, lse, d_o, dq, dk, dv)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with _on(q):
        st = _stream(stream, q.device)
        handles = []
        for ev in (ev_main_begin, ev_main_end):
            if ev is None or isinstance(ev, int):
                handles.append(_vp(ev))
            else:
                if not ev.cuda_event:  # torch creates its event at the first record
                    import torch
                    ev.record(torch.cuda.current_stream(q.device))
                handles.append(_vp(ev.cuda_event))
        _check(_c_bwd_timed(plan.handle, _dtype_code(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o),
                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), ws_bytes, T, Hq, Hkv, D,
                            float(softmax_scale), 1 if deterministic else 0, handles[0], handles[1], _ptr(d_status),
                            st), "sp_tree_attn_bwd_timed")


def sp_tree_attn_bwd_noalloc(plan: Plan, q, k, v, o, lse, d_o, dq, dk, dv, softmax_scale: float,
                             d_status=None, stream=None):
    """sp_tree_attn_bwd backed by the library's fixed device scratch (no workspace)."""
    _need_cuda(q, k, v, o, lse, d_o, dq, dk, dv, d_status)
    _need_status(d_status)
    T, Hq, Hkv, D = _check_bwd_shapes(q, k, v, o, lse, d_o, dq, dk, dv)
    with _on(q):
        _check(_c_bwd_noalloc(plan.handle, _dtype_code(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                              _ptr(d_o), _ptr(dq), _ptr(dk), _ptr(dv), T, Hq, Hkv, D, float(softmax_scale),
                              _ptr(d_status), _stream(stream, q.device)), "sp_tree_attn_bwd_noalloc")


def sp_edge_gather(hidden, idx, out, d_status=None, stream=None):
    _need_cuda(hidden, idx, out, d_status)
    _need_status(d_status)
    import torch
    if idx.dtype != torch.int32:
        raise ValueError("edge indices must be int32")
    T, Hd = hidden.shape
    E = idx.shape[0]
    if tuple(out.shape) != (E, Hd) or out.dtype != hidden.dtype:
        raise ValueError("shape or dtype mismatch")
    with _on(hidden):
        _check(_c_gather(_dtype_code(hidden), _ptr(hidden), T, Hd, _ptr(idx), E, _ptr(out), _ptr(d_status),
                         _stream(stream, hidden.device)), "sp_edge_gather")


def sp_edge_gather_bwd_workspace_bytes(T: int, E: int) -> int:
    return int(_c_gather_bwd_ws(T, E))


def sp_edge_gather_bwd(grad_out, idx, grad_hidden, workspace, d_status=None, stream=None):
    _need_cuda(grad_out, idx, grad_hidden, workspace, d_status)
    _need_status(d_status)
    import torch
    if idx.dtype != torch.int32:
        raise ValueError("edge indices must be int32")
    E, Hd = grad_out.shape
    T = grad_hidden.shape[0]
    if tuple(grad_hidden.shape) != (T, Hd) or grad_hidden.dtype != grad_out.dtype or idx.shape[0] != E:
        raise ValueError("shape or dtype mismatch")
    ws = workspace.numel() * workspace.element_size()
    with _on(grad_hidden):
        _check(_c_gather_bwd(_dtype_code(grad_out), _ptr(grad_out), E, Hd, _ptr(idx), T, _ptr(grad_hidden),
                             _ptr(workspace), ws, _ptr(d_status), _stream(stream, grad_hidden.device)),
               "sp_edge_gather_bwd")


def sp_edge_logprob_workspace_bytes(E: int, V: int) -> int:
    return int(_c_lmh_ws(E, V))


def sp_edge_logprob(hidden_sel, weight, labels, logprob, lse, workspace, d_status=None, stream=None):
    _need_cuda(hidden_sel, weight, labels, logprob, lse, workspace, d_status)
    _need_status(d_status)
    import torch
    if labels.dtype != torch.int32 or logprob.dtype != torch.float32 or lse.dtype != torch.float32:
        raise ValueError("labels must be int32, logprob and lse float32")
    E, Hd = hidden_sel.shape
    V = weight.shape[0]
    if weight.shape[1] != Hd or labels.shape[0] != E or logprob.shape[0] != E or lse.shape[0] != E:
        raise ValueError("shape mismatch")
    ws = workspace.numel() * workspace.element_size()
    with _on(weight):
        _check(_c_lmh(_dtype_code(hidden_sel), _ptr(hidden_sel), E, Hd, _ptr(weight), V, _ptr(labels),
                      _ptr(logprob), _ptr(lse), _ptr(workspace), ws, _ptr(d_status), _stream(stream, weight.device)),
               "sp_edge_logprob")


def sp_edge_logprob_bwd_workspace_bytes(E: int, V: int) -> int:
    return int(_c_lmh_bwd_ws(E, V))


def sp_edge_logprob_bwd(hidden_sel, weight, labels, lse, grad_logprob, d_hidden_sel, d_weight, workspace,
                        d_status=None, stream=None):
    _need_cuda(hidden_sel, weight, labels, lse, grad_logprob, d_hidden_sel, d_weight, workspace, d_status)
    _need_status(d_status)
    import torch
    E, Hd = hidden_sel.shape
    V = weight.shape[0]
    for t, shape in ((d_hidden_sel, (E, Hd)), (d_weight, (V, Hd))):
        if t is not None and (tuple(t.shape) != shape or t.dtype != torch.float32):
            raise ValueError("gradient outputs must be float32 [E, Hd] and [V, Hd]")
    if labels.dtype != torch.int32 or lse.dtype != torch.float32 or grad_logprob.dtype != torch.float32:
        raise ValueError("labels int32, lse and grad_logprob float32")
    ws = workspace.numel() * workspace.element_size()
    with _on(weight):
        _check(_c_lmh_bwd(_dtype_code(hidden_sel), _ptr(hidden_sel), E, Hd, _ptr(weight), V, _ptr(labels),
                          _ptr(lse), _ptr(grad_logprob), _ptr(d_hidden_sel), _ptr(d_weight), _ptr(workspace), ws,
                          _ptr(d_status), _stream(stream, weight.device)), "sp_edge_logprob_bwd")


def sp_debug_wait_timeout(spin_limit: int, d_status, stream=None):
    _need_cuda(d_status)
    _need_status(d_status)
    with _on(d_status):
        _check(_c_wait_timeout(int(spin_limit), _ptr(d_status), _stream(stream, d_status.device)),
               "sp_debug_wait_timeout")


CLOCK_FORWARD, CLOCK_KEY_BLOCKS, CLOCK_QUERY_TILES = 1, 2, 3


def sp_debug_cta_clock(kernel: int, buffer=None):
    """Record per-CTA start/end times of one tensor-core kernel's later launches into ``buffer`` (a CUDA
    uint64 tensor of shape [n, 4]: start ns, end ns, SM id, 0 per CTA); ``kernel`` 0 or no buffer: off."""
    import torch
    if buffer is None or kernel == 0:
        _check(_c_cta_clock(0, None, 0), "sp_debug_cta_clock")
        return
    _need_cuda(buffer)
    if buffer.dtype not in (torch.int64, torch.uint64) or buffer.dim() != 2 or buffer.shape[1] != 4:
        raise ValueError("buffer must be an int64 CUDA tensor of shape [n, 4]")
    _check(_c_cta_clock(int(kernel), _ptr(buffer), int(buffer.shape[0])), "sp_debug_cta_clock")


# ------------------------------------------------------------ conveniences
# Thin allocating wrappers over the entry points above (torch.empty only).

def sp_fragment_plan(seg_start, seg_len, parent, depth, max_tokens: int) -> dict:
    """Bounded fragments of a tree: the sp_fragment_view tables as numpy arrays (the handle is freed)."""
    arrs = [np.ascontiguousarray(np.asarray(a, dtype=np.int32)) for a in (seg_start, seg_len, parent, depth)]
    n = int(arrs[0].shape[0])
    total = int(arrs[1].astype(np.int64).sum()) if n else 0
    desc = _TreeDesc(n, total, *[a.ctypes.data_as(_i32p) for a in arrs])
    h = ctypes.c_void_p()
    _check(_c_frag_plan(ctypes.byref(desc), int(max_tokens), ctypes.byref(h)), "sp_fragment_plan")
    try:
        info = _FragInfo()
        _check(_c_frag_view(h, ctypes.byref(info)), "sp_fragment_view")
        nf, ne = info.num_fragments, info.num_entries

        def arr(p, k):
            return np.ctypeslib.as_array(p, shape=(k,)).copy() if k else np.zeros(0, dtype=np.int32)

        return {"num_fragments": nf, "physical_tokens": int(info.physical_tokens),
                "fragment_tokens": int(info.fragment_tokens), "offsets": arr(info.offsets, nf + 1),
                "tokens": arr(info.tokens, nf), "seg": arr(info.seg, ne), "owned": arr(info.owned, ne),
                "local_parent": arr(info.local_parent, ne), "local_start": arr(info.local_start, ne)}
    finally:
        _c_frag_destroy(h)


def fragment_plan(tree, max_tokens: int) -> dict:
    """sp_fragment_plan for any object with seg_start/seg_len/parent/depth arrays."""
    return sp_fragment_plan(tree.seg_start, tree.seg_len, tree.parent, tree.depth, max_tokens)


def fragment_tree(frag: dict, f: int, tree):
    """Fragment f's own packed tree: (seg_start, seg_len, parent, depth, segments, owned)."""
    a, b = int(frag["offsets"][f]), int(frag["offsets"][f + 1])
    segs = frag["seg"][a:b]
    return (frag["local_start"][a:b].copy(), np.asarray(tree.seg_len)[segs].astype(np.int32),
            frag["local_parent"][a:b].copy(), np.asarray(tree.depth)[segs].astype(np.int32), segs.copy(),
            frag["owned"][a:b].copy())


def fragment_tokens(frag: dict, f: int, tree):
    """(token index [n], owned [n] bool) of fragment f: row i of the fragment's packed buffer is row
    token_index[i] of the whole tree's; owned marks the tokens whose outputs and loss this fragment owns."""
    a, b = int(frag["offsets"][f]), int(frag["offsets"][f + 1])
    idx, own = [], []
    for s_, o_ in zip(frag["seg"][a:b], frag["owned"][a:b]):
        start, n = int(tree.seg_start[s_]), int(tree.seg_len[s_])
        idx.append(np.arange(start, start + n, dtype=np.int64))
        own.append(np.full(n, bool(o_)))
    if not idx:
        return np.zeros(0, dtype=np.int64), np.zeros(0, dtype=bool)
    return np.concatenate(idx), np.concatenate(own)


def tree_plan(tree, tile_tokens: int, kv_block: int = 128, order: int = 0, upload: bool = True) -> Plan:
    """Plan from any object with seg_start/seg_len/parent/depth arrays."""
    p = sp_tree_plan(tree.seg_start, tree.seg_len, tree.parent, tree.depth, tile_tokens, kv_block, order)
    if upload:
        sp_plan_upload(p)
    return p


def tree_attn_fwd(plan: Plan, q, k, v, softmax_scale: float, d_status=None):
    import torch
    o = torch.empty_like(q)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    sp_tree_attn_fwd(plan, q, k, v, o, lse, softmax_scale, d_status)
    return o, lse


def bwd_workspace(q) -> "torch.Tensor":
    import torch
    n = sp_tree_attn_bwd_workspace_bytes(_dtype_code(q), q.shape[0], q.shape[1], q.shape[2])
    return torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)


def tree_attn_bwd(plan: Plan, q, k, v, o, lse, d_o, softmax_scale: float, workspace=None, d_status=None,
                  deterministic: bool = False):
    import torch
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = bwd_workspace(q) if workspace is None else workspace
    fn = sp_tree_attn_bwd_deterministic if deterministic else sp_tree_attn_bwd
    fn(plan, q, k, v, o, lse, d_o, dq, dk, dv, ws, softmax_scale, d_status)
    return dq, dk, dv


def edge_logprob(hidden_sel, weight, labels, d_status=None):
    """(logprob [E], lse [E]) of each action's label through the vocabulary head."""
    import torch
    E = hidden_sel.shape[0]
    lp = torch.empty(E, dtype=torch.float32, device=hidden_sel.device)
    lse = torch.empty(E, dtype=torch.float32, device=hidden_sel.device)
    ws = torch.empty(max(256, sp_edge_logprob_workspace_bytes(E, weight.shape[0])), dtype=torch.uint8,
                     device=hidden_sel.device)
    sp_edge_logprob(hidden_sel, weight, labels, lp, lse, ws, d_status)
    return lp, lse


def edge_logprob_bwd(hidden_sel, weight, labels, lse, grad_logprob, d_status=None):
    """(d_hidden_sel [E, Hd], d_weight [V, Hd]) in fp32."""
    import torch
    E, Hd = hidden_sel.shape
    V = weight.shape[0]
    dh = torch.empty((E, Hd), dtype=torch.float32, device=hidden_sel.device)
    dw = torch.empty((V, Hd), dtype=torch.float32, device=hidden_sel.device)
    ws = torch.empty(max(256, sp_edge_logprob_bwd_workspace_bytes(E, V)), dtype=torch.uint8, device=hidden_sel.device)
    sp_edge_logprob_bwd(hidden_sel, weight, labels, lse, grad_logprob, dh, dw, ws, d_status)
    return dh, dw


def edge_gather_bwd(grad_out, idx, num_tokens: int, d_status=None):
    import torch
    gh = torch.empty((num_tokens, grad_out.shape[1]), dtype=grad_out.dtype, device=grad_out.device)
    ws = torch.empty(max(16, sp_edge_gather_bwd_workspace_bytes(num_tokens, idx.shape[0])), dtype=torch.uint8,
                     device=grad_out.device)
    sp_edge_gather_bwd(grad_out, idx, gh, ws, d_status)
    return gh


def edge_gather(hidden, idx, d_status=None):
    import torch
    out = torch.empty((idx.shape[0], hidden.shape[1]), dtype=hidden.dtype, device=hidden.device)
    sp_edge_gather(hidden, idx, out, d_status)
    return out
