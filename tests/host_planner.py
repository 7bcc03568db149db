"""A host-only build of the library's planners, for CPU tests.

``plan.cpp`` and ``fragments.cpp`` (optionally one of them with a planted
change) are compiled with g++ together with ``tests/c/planner_shim.cpp`` into a
small shared library: no CUDA.  ``Host`` calls it through ctypes: the plan
tables, the tables the kernels read (built as the first upload builds them) and
the fragment planner.
"""
import ctypes
import os
import subprocess

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "shared_prefix_causal_gb300", "csrc")
SHIM = os.path.join(ROOT, "tests", "c", "planner_shim.cpp")
SOURCES = ("plan.cpp", "fragments.cpp")

class _Desc(ctypes.Structure):
    _fields_ = [("num_segments", ctypes.c_int32), ("total_tokens", ctypes.c_int32)] + \
               [(n, ctypes.POINTER(ctypes.c_int32)) for n in ("seg_start", "seg_len", "parent", "depth")]


class _FragInfo(ctypes.Structure):
    _fields_ = [("num_fragments", ctypes.c_int32), ("num_entries", ctypes.c_int32),
                ("physical_tokens", ctypes.c_int64), ("fragment_tokens", ctypes.c_int64)] + \
               [(n, ctypes.POINTER(ctypes.c_int32)) for n in ("offsets", "tokens", "seg", "owned", "local_parent",
                                                              "local_start")]


class Host:
    """ctypes view of one host-only build."""

    def __init__(self, path):
        self.lib = ctypes.CDLL(path)
        self.lib.shim_plan.restype = ctypes.c_void_p
        self.lib.shim_plan.argtypes = [ctypes.POINTER(_Desc), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.POINTER(ctypes.c_int32)]
        self.lib.shim_rows.restype = ctypes.c_int32
        self.lib.shim_rows.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.POINTER(ctypes.c_int32))]
        self.lib.shim_free.argtypes = [ctypes.c_void_p]
        self.lib.shim_device_tables.argtypes = [ctypes.c_void_p]
        self.lib.shim_merge_runs.restype = ctypes.c_int32
        self.lib.shim_merge_runs.argtypes = [ctypes.POINTER(ctypes.c_int32)] * 2 + \
            [ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32]
        self.lib.shim_bwd_run_sum.restype = ctypes.c_int64
        self.lib.shim_bwd_run_sum.argtypes = [ctypes.c_void_p]
        self.lib.shim_bwd_run_max.restype = ctypes.c_int32
        self.lib.shim_bwd_run_max.argtypes = [ctypes.c_void_p]
        self.lib.shim_bwdm_run_sum.restype = ctypes.c_int64
        self.lib.shim_bwdm_run_sum.argtypes = [ctypes.c_void_p]
        self.lib.shim_bwdm_run_max.restype = ctypes.c_int32
        self.lib.shim_bwdm_run_max.argtypes = [ctypes.c_void_p]
        self.lib.sp_fragment_plan.argtypes = [ctypes.POINTER(_Desc), ctypes.c_int64, ctypes.POINTER(ctypes.c_void_p)]
        self.lib.sp_fragment_view.argtypes = [ctypes.c_void_p, ctypes.POINTER(_FragInfo)]
        self.lib.sp_fragment_destroy.argtypes = [ctypes.c_void_p]

    @staticmethod
    def _desc(st, ln, par, dep, total=None):
        arrs = [np.ascontiguousarray(np.asarray(a, dtype=np.int32)) for a in (st, ln, par, dep)]
        total = int(arrs[1].sum()) if total is None else total
        return _Desc(len(arrs[0]), total, *[a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) for a in arrs]), arrs

    def _rows(self, h, which, w):
        ptr = ctypes.POINTER(ctypes.c_int32)()
        n = self.lib.shim_rows(h, which, ctypes.byref(ptr))
        return np.ctypeslib.as_array(ptr, shape=(n * w,)).reshape(n, w).copy() if n else np.zeros((0, w), np.int32)

    def plan(self, st, ln, par, dep, tile, kvb, order, total=None):
        """(tiles, ranges, bwd), or the status of a refused call."""
        d, keep = self._desc(st, ln, par, dep, total)
        rc = ctypes.c_int32()
        h = self.lib.shim_plan(ctypes.byref(d), tile, kvb, order, ctypes.byref(rc))
        if rc.value:
            return rc.value
        out = tuple(self._rows(h, which, w) for which, w in ((0, 5), (1, 2), (2, 5)))
        self.lib.shim_free(h)
        return out

    def device_tables(self, st, ln, par, dep, tile, kvb, order):
        """The plan and the tables its first upload builds: a dict of tiles, ranges, bwd, pairs, pblk,
        bwd_sched, quads, qblk, bwd_merged, key_end, run_sum, run_max, runm_sum and runm_max, or the
        status of a refused call."""
        d, keep = self._desc(st, ln, par, dep)
        rc = ctypes.c_int32()
        h = self.lib.shim_plan(ctypes.byref(d), tile, kvb, order, ctypes.byref(rc))
        if rc.value:
            return rc.value
        self.lib.shim_device_tables(h)
        names = ("tiles", "ranges", "bwd", "pairs", "pblk", "bwd_sched", "quads", "qblk", "bwd_merged", "key_end")
        out = {n: self._rows(h, i, w) for i, (n, w) in enumerate(zip(names, (5, 2, 5, 4, 8, 5, 6, 8, 5, 1)))}
        out["key_end"] = out["key_end"].reshape(-1)
        out["run_sum"], out["run_max"] = int(self.lib.shim_bwd_run_sum(h)), int(self.lib.shim_bwd_run_max(h))
        out["runm_sum"], out["runm_max"] = int(self.lib.shim_bwdm_run_sum(h)), int(self.lib.shim_bwdm_run_max(h))
        self.lib.shim_free(h)
        return out

    def merge_runs(self, lists, block_keys):
        """The planner's run merge on arbitrary lists: lists[i] = [(kb, nb, end, causal), ...] for slots
        0..3; returns the entries [n][8]."""
        flat = np.array([x for l in lists for r in l for x in r] or [0], dtype=np.int32)
        counts = np.array([len(l) for l in lists], dtype=np.int32)
        cap = sum(r[1] for l in lists for r in l) + 1
        out = np.zeros(8 * cap, dtype=np.int32)
        p32 = ctypes.POINTER(ctypes.c_int32)
        n = self.lib.shim_merge_runs(flat.ctypes.data_as(p32), counts.ctypes.data_as(p32), block_keys,
                                     out.ctypes.data_as(p32), cap)
        return out[:8 * n].reshape(n, 8)

    def fragments(self, st, ln, par, dep, cap):
        d, keep = self._desc(st, ln, par, dep)
        h = ctypes.c_void_p()
        rc = self.lib.sp_fragment_plan(ctypes.byref(d), cap, ctypes.byref(h))
        if rc:
            return rc
        info = _FragInfo()
        assert self.lib.sp_fragment_view(h, ctypes.byref(info)) == 0
        get = lambda p, n: np.ctypeslib.as_array(p, shape=(n,)).copy() if n else np.zeros(0, np.int32)  # noqa: E731
        ne, nf = info.num_entries, info.num_fragments
        out = {k: get(getattr(info, k), ne) for k in ("seg", "owned", "local_parent", "local_start")}
        out["offsets"], out["tokens"] = get(info.offsets, nf + 1), get(info.tokens, nf)
        self.lib.sp_fragment_destroy(h)
        return out


_CXX = ["g++", "-std=c++17", "-O0", "-fPIC", "-fvisibility=hidden", "-I", CSRC]


def compile_object(src, obj):
    subprocess.run(_CXX + ["-c", str(src), "-o", str(obj)], check=True, capture_output=True, text=True)
    return str(obj)


def original_objects(d):
    """The unchanged sources and the shim compiled into ``d`` (a pathlib directory)."""
    objs = {f: compile_object(os.path.join(CSRC, f), d / (f + ".o")) for f in SOURCES}
    objs["shim"] = compile_object(SHIM, d / "shim.o")
    return objs


def build_host_library(objs, d, mutant=None):
    """A host-only library: the original objects, with the mutated file (if any) recompiled.

    ``mutant`` is (file, text, replacement, ...): the text must occur exactly once in the file."""
    d.mkdir()
    parts = dict(objs)
    if mutant:
        f, old, new = mutant[:3]
        text = open(os.path.join(CSRC, f), encoding="utf-8").read()
        assert text.count(old) == 1, f"{f}: the planted text must occur exactly once: {old!r}"
        (d / f).write_text(text.replace(old, new))
        parts[f] = compile_object(d / f, d / (f + ".o"))
    out = str(d / "libhost.so")
    subprocess.run(["g++", "-shared", *parts.values(), "-o", out], check=True, capture_output=True, text=True)
    return Host(out)


