"""Benchmark: shared-prefix tree attention forward + backward on one GB300.

One step = the whole hot path over one batch: tree attention forward,
backward (which includes its preprocess and dQ conversion kernels) and the
sampled-edge gather, on the seeded synthetic agent-call tree (65,536 tokens,
32 query heads, 8 KV heads, head_dim 128, bf16) unless ``--config`` names
another workload.  The plan is built once per tree; the end-to-end figure
rebuilds and uploads it every step.

Prints one JSON line.  ``value`` is useful (ancestor-masked) attention
TFLOP/s with inputs resident in HBM: 4*D*Hq*pairs forward plus 10*D*Hq*pairs
backward per step, where pairs counts only visible (query, key) pairs.

``--impl reference`` times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload per step).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "tree-attn fwd+bwd useful TFLOP/s and tokens/s at 1 GB300; % of BF16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# kernels the library launches per call (fwd; bwd = preprocess, main, dQ; gather)
LAUNCHES_PER_STEP = {"fwd": 1, "bwd": 3, "gather": 1}
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of each tensor-core kernel,
# from one single-pass ncu capture of this bench on a GB300 (one launch of the kernel, warm-up step 2),
# keyed by workload, with a digest of the code (comments stripped) that defines the kernel and its
# schedule: a figure whose code has changed since the capture is reported as null.  "file:function"
# takes one function of a file: the planner's schedule builders decide the launch order, while the
# canonical plan they start from is fixed bit for bit by the planner's tests.
CSRC = os.path.join(ROOT, "shared_prefix_causal_gb300", "csrc")
TRAFFIC_SOURCES = {
    "fwd_tc_kernel": ("attn_fwd_sm103a.cu", "sm103_ptx.cuh", "pipeline.cuh", "plan.cpp:build_pairs",
                      "plan.cpp:tile_runs", "plan.cpp:merge_runs"),
    "bwd_tc_kernel": ("attn_bwd_sm103a.cu", "sm103_ptx.cuh", "pipeline.cuh", "plan.cpp:build_bwd_schedule",
                      "plan.cpp:build_bwd_merged"),
}
# DRAM bytes (read + write) of one launch, from an ncu capture of one launch of the kernel on the
# named workload (dram__bytes_read.sum + dram__bytes_write.sum), with the digest of the code that
# decides that traffic; the units are query heads x useful pairs of that workload.
MEASURED_TRAFFIC = {
    "tiny": {"units": 26252,
             "fwd_tc_kernel": (195840 + 0, "6551394c778f6917"),
             "bwd_tc_kernel": (346624 + 0, "2a5e1bb63e8773c4")},
    "star": {"units": 506117152,
             "fwd_tc_kernel": (94208000 + 27344384, "6551394c778f6917"),
             "bwd_tc_kernel": (345844224 + 142123520, "2a5e1bb63e8773c4")},
    "agent_small": {"units": 2424419552,
                    "fwd_tc_kernel": (202022144 + 100264960, "6551394c778f6917"),
                    "bwd_tc_kernel": (2019589120 + 981808384, "2a5e1bb63e8773c4")},
    "long_small": {"units": 8211399552,
                   "fwd_tc_kernel": (336584704 + 232509952, "6551394c778f6917"),
                   "bwd_tc_kernel": (9595139840 + 5118466560, "2a5e1bb63e8773c4")},
    "forest_small": {"units": 3793239488,
                     "fwd_tc_kernel": (499851008 + 303153920, "6551394c778f6917"),
                     "bwd_tc_kernel": (3449080064 + 1793794560, "2a5e1bb63e8773c4")},
}
# Full-size workloads are not captured with more than the launch time: their traffic is the reduced
# workload's of the same shape, scaled by the ratio of units (query heads x useful pairs).
TRAFFIC_SCALED_FROM = {"agent": "agent_small", "long": "long_small", "forest": "forest_small"}


# ------------------------------------------------------------------ helpers

def useful_pairs(tree) -> int:
    """Visible (query, key) pairs: sum over segments of len*len(ancestors) + len*(len+1)/2."""
    anc = np.zeros(tree.num_segments, dtype=np.int64)
    total = 0
    for s in range(tree.num_segments):
        p = int(tree.parent[s])
        if p >= 0:
            anc[s] = anc[p] + int(tree.seg_len[p])
        n = int(tree.seg_len[s])
        total += n * int(anc[s]) + n * (n + 1) // 2
    return total


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments, blank lines or trailing blanks (comments do not change a kernel)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def _function_text(code: str, name: str) -> str:
    """The definition of function ``name`` (signature line to closing brace) in comment-free code."""
    import re
    m = re.search(r"^[^\n;{}]*\b" + re.escape(name) + r"\s*\([^;{]*\)\s*\{", code, flags=re.M)
    if m is None:
        raise KeyError(name)
    depth, i = 1, m.end()
    while depth:
        depth += {"{": 1, "}": -1}.get(code[i], 0)
        i += 1
    return code[m.start():i]


def sources_digest(kernel: str) -> str:
    import hashlib
    m = hashlib.sha256()
    for f in TRAFFIC_SOURCES[kernel]:
        path, _, func = f.partition(":")
        with open(os.path.join(CSRC, path), encoding="utf-8") as fh:
            code = _code_only(fh.read())
        m.update((_function_text(code, func) if func else code).encode())
    return m.hexdigest()[:16]


def measured_traffic(config: str, kernel: str, units: int):
    """(DRAM bytes per launch, how they were obtained), or (None, why) if absent or stale."""
    src = config if config in MEASURED_TRAFFIC else TRAFFIC_SCALED_FROM.get(config)
    entry = MEASURED_TRAFFIC.get(src, {}).get(kernel)
    if entry is None:
        return None, "no capture"
    if sources_digest(kernel) != entry[1]:
        return None, "capture predates the kernel's current code"
    if src == config:
        return int(entry[0]), "ncu capture of one launch on this workload"
    scale = units / MEASURED_TRAFFIC[src]["units"]
    return int(round(entry[0] * scale)), f"ncu capture of one launch on {src}, scaled by units x{scale:.3f}"


def tile_efficiency(spc, plan, G: int, pairs: int) -> dict:
    """Useful pairs over the pairs the kernels compute (full 128-key blocks of 128-row tiles
    forward; 64-row query blocks against the backward's merged 128-key blocks), per query head."""
    v = spc.sp_plan_view(plan)
    tt = int(v["tile_tokens"])
    fwd = 0
    for _, q0, q1, rb, rc in v["tiles"].tolist():
        nb = sum((e - a + 127) // 128 for a, e in v["ranges"][rb:rb + rc].tolist())
        fwd += nb * 128 * tt
    tpb = 64 // G
    bwd = sum(((q1 - q0 + tpb - 1) // tpb) * tpb * 128
              for _, _, _, q0, q1 in spc.sp_plan_bwd_blocks(plan)["rows"].tolist())
    return {"fwd": round(pairs / max(fwd, 1), 4), "bwd": round(pairs / max(bwd, 1), 4)}


def load_peaks(path=None):
    path = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def _number(x):
    """A plain number, or one held under value/median/mean of a small record."""
    if isinstance(x, (int, float)) and not isinstance(x, bool):
        return float(x)
    if isinstance(x, dict):
        for k in ("value", "median", "mean"):
            if isinstance(x.get(k), (int, float)) and not isinstance(x.get(k), bool):
                return float(x[k])
    return None


def _peak_value(peaks, *keys):
    """The first of ``keys`` found with a number, at the top level of ``peaks`` or one level down."""
    if not isinstance(peaks, dict):
        return None
    for k in keys:
        for d in [peaks] + [v for v in peaks.values() if isinstance(v, dict)]:
            if k in d and _number(d[k]) is not None:
                return _number(d[k])
    return None


PEAK_KEYS = {"burst": ("bf16_tflops", "bf16_tflops_burst"), "sustained": ("bf16_tflops_sustained",),
             "hbm": ("hbm_gbs",)}


def resolve_peaks(peaks, source):
    """{name: (value, "measured" | "fallback")}: the measured figure where the file has a positive one,
    else the fallback figure."""
    out = {}
    for name, keys in PEAK_KEYS.items():
        v = _peak_value(peaks, *keys) if source == "measured" else None
        out[name] = (v, "measured") if v is not None and v > 0 else (_peak_value(FALLBACK_PEAKS, *keys), "fallback")
    return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.window = None

    def mark(self, begin: float, end: float):
        """Wall-clock bounds of the timed region: only samples inside it are kept."""
        self.window = (begin, end)

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        import datetime
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    clk, cmax = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    ts = None  # unparsable timestamp: keep the sample
                if self.window and ts is not None and not (self.window[0] - 0.05 <= ts <= self.window[1] + 0.05):
                    continue
                sm.append(clk)
                smax.append(cmax)
                for n, val in zip(names, parts[6:10]):
                    if val.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------- oracle (CPU) leg

def _subtree_of_leaves(tree, leaves):
    """Re-pack the union of some root-to-leaf paths as its own preorder tree.

    Returns (tree, token_index) where token_index maps new tokens to old."""
    from oracle import tree as OT
    keep = set()
    for l in leaves:
        keep.update(OT.ancestors(tree.parent, l))
        keep.add(l)
    order = sorted(keep)  # preorder is preserved by index order
    newid = {s: i for i, s in enumerate(order)}
    lens = [int(tree.seg_len[s]) for s in order]
    pars = [newid[int(tree.parent[s])] if int(tree.parent[s]) >= 0 else -1 for s in order]
    tok = np.concatenate([np.arange(int(tree.seg_start[s]), int(tree.seg_start[s]) + int(tree.seg_len[s]))
                          for s in order])
    return W.tree_from_preorder(lens, pars), tok


def oracle_sample_plan(w, flop_budget: float):
    """Root-to-leaf paths of the workload, shortest first, while their
    unrolled fp64 cost (KV group 0) stays within ``flop_budget``; at least one."""
    from oracle import tree as OT
    t = w.tree
    G = w.hq // w.hkv
    leaves = OT.leaves(t.parent)
    plen = {l: len(OT.path_tokens(t.seg_start, t.seg_len, t.parent, l)) for l in leaves}
    chosen, cost = [], 0.0
    for l in sorted(leaves, key=lambda l: (plen[l], l)):
        c = 14.0 * w.head_dim * G * plen[l] * plen[l] / 2
        if chosen and cost + c > flop_budget:
            break
        chosen.append(l)
        cost += c
    return sorted(chosen)


def oracle_child(spec: dict):
    """Runs in a fresh interpreter: times the oracle on one sample."""
    from oracle import attention as A
    w = W.get(spec["config"])
    sub, tok = _subtree_of_leaves(w.tree, spec["leaves"])
    x = W.draw_tensors(w, "bf16")
    G = w.hq // w.hkv
    q = x["q"][tok][:, :G].float().numpy()
    k = x["k"][tok][:, :1].float().numpy()
    v = x["v"][tok][:, :1].float().numpy()
    do = x["do"][tok][:, :G].float().numpy()
    args = (sub.seg_start, sub.seg_len, sub.parent, w.softmax_scale)
    times = []
    for _ in range(spec.get("reps", 1)):
        t0 = time.perf_counter()
        A.tree_forward(q, k, v, *args)
        A.tree_backward(q, k, v, do, *args)
        times.append(time.perf_counter() - t0)
    pairs = useful_pairs(sub)
    flops = 14.0 * w.head_dim * G * pairs
    print(json.dumps({"times": times, "useful_flops": flops, "tokens": int(sub.total_tokens),
                      "paths": len(spec["leaves"])}))


def run_oracle_sample(w, flop_budget: float, reps: int = 1):
    leaves = oracle_sample_plan(w, flop_budget)
    cores = len(os.sched_getaffinity(0))
    env = dict(os.environ)
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    spec = {"config": w.name, "leaves": [int(l) for l in leaves], "reps": reps}
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--_oracle-child", json.dumps(spec)],
                       capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed: " + r.stderr[-2000:])
    out = json.loads(r.stdout.strip().splitlines()[-1])
    out["cores"] = cores
    out["sample"] = (f"KV head 0 ({w.hq // w.hkv} query heads) over the {len(leaves)} shortest root-to-leaf "
                     f"paths ({out['tokens']} physical tokens of {w.T}), fwd+bwd, fp64 leaf-unrolled "
                     f"NumPy, {cores} BLAS threads")
    return out


# --------------------------------------------------------------- GPU leg

def max_over_ranks(value: float, device=None) -> float:
    """The largest value any rank holds (the job's time is its slowest rank's).

    Replicas only: this timing reduction is the one collective; no data moves
    between ranks."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, ranks: int, slowest_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest time."""
    return units_per_rank * ranks / (slowest_ms * 1e-3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_gpu(args):
    import torch

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    import shared_prefix_causal_gb300 as spc

    w = W.get(args.config)
    G = w.hq // w.hkv
    T, D = w.T, w.head_dim
    x = W.draw_tensors(w, "bf16", with_hidden=w.hidden_dim is not None)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    hidden = x["hidden"].to(dev) if "hidden" in x else None
    idx = torch.from_numpy(w.edge_idx).to(dev) if w.edge_idx is not None else None
    scale = w.softmax_scale

    t0 = time.perf_counter()
    plan = spc.tree_plan(w.tree, 128 // G, 128, 0, upload=False)
    plan_ms = (time.perf_counter() - t0) * 1e3
    spc.sp_plan_upload(plan)
    o = torch.empty_like(q)
    lse = torch.empty((w.hq, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_buf = spc.bwd_workspace(q)
    gathered = torch.empty((idx.shape[0], hidden.shape[1]), dtype=hidden.dtype, device=dev) \
        if hidden is not None else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        spc.sp_tree_attn_fwd(plan, q, k, v, o, lse, scale, status)
        if evs:
            evs[1].record(stream)
            # the same backward call, with two more events recorded around its main kernel
            spc.sp_tree_attn_bwd_timed(plan, q, k, v, o, lse, do, dq, dk, dv, ws_buf, scale, False, evs[4], evs[5],
                                       status)
            evs[2].record(stream)
        else:
            spc.sp_tree_attn_bwd(plan, q, k, v, o, lse, do, dq, dk, dv, ws_buf, scale, status)
        if hidden is not None:
            spc.sp_edge_gather(hidden, idx, gathered, status)
        if evs:
            evs[3].record(stream)

    clocks = ClockSampler(dev.index)
    clocks.start()  # running before the timed region: nvidia-smi takes a moment to start sampling
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item()} during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for e in evs:  # torch creates an event's handle at its first record
        for x_ in e:
            x_.record(stream)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    stop.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(wall0, time.time())
    clk = clocks.stop()
    if ws > 1:
        torch.distributed.barrier()
    total_ms = start.elapsed_time(stop)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    gat_ms = [e[2].elapsed_time(e[3]) for e in evs]
    main_ms = [e[4].elapsed_time(e[5]) for e in evs]  # the backward's main kernel alone
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item()} in the timed region")
    if ws > 1:
        total_ms = max_over_ranks(total_ms, dev)

    pairs = useful_pairs(w.tree)
    f_fwd = 4.0 * D * w.hq * pairs
    f_bwd = 10.0 * D * w.hq * pairs
    traffic_fwd = measured_traffic(args.config, "fwd_tc_kernel", w.hq * pairs)
    traffic_bwd = measured_traffic(args.config, "bwd_tc_kernel", w.hq * pairs)
    ms_step = total_ms / args.steps
    value = job_throughput(f_fwd + f_bwd, ws, ms_step) / 1e12
    pk = resolve_peaks(*load_peaks())
    (p_burst, src_burst), (p_sust, src_sust), (p_hbm, _) = pk["burst"], pk["sustained"], pk["hbm"]
    med_fwd, med_bwd = statistics.median(fwd_ms), statistics.median(bwd_ms)
    fwd_tflops = f_fwd / (med_fwd * 1e-3) / 1e12
    bwd_tflops = f_bwd / (med_bwd * 1e-3) / 1e12
    mean_bwd = statistics.mean(bwd_ms)
    mean_main = statistics.mean(main_ms)
    mean_fwd = statistics.mean(fwd_ms)
    # one cold-L2 step: a 256 MiB scrub written just before it
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0))
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cold_ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for x_ in cold_ev:
        x_.record(stream)
    scrub.fill_(1)
    step(cold_ev)
    torch.cuda.synchronize(dev)
    del scrub
    cold = {"fwd_ms": round(cold_ev[0].elapsed_time(cold_ev[1]), 4),
            "bwd_ms": round(cold_ev[1].elapsed_time(cold_ev[2]), 4), "scrub_bytes": 256 << 20}
    e2e = run_e2e(args, spc, w, x, dev, f_fwd + f_bwd) if rank == 0 and not args.no_e2e else None
    det = run_deterministic_bwd(args, spc, plan, q, k, v, o, lse, do, dq, dk, dv, ws_buf, scale, status, dev, f_bwd,
                                p_burst)
    paired = run_paired_fwd(args, spc, plan, q, k, v, o, lse, scale, status, dev, f_fwd, p_burst)
    lm_head = run_lm_head(args, spc, w, gathered, idx, dev, p_burst, p_sust) \
        if gathered is not None and not args.no_lm_head else None

    # compulsory bytes: every input read once, every output written once
    algo_fwd = T * (2 * w.hq * D * 2 + 2 * w.hkv * D * 2 + 4 * w.hq)
    algo_bwd = T * (4 * w.hq * D * 2 + 4 * w.hkv * D * 2 + 8 * w.hq)
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; inputs drawn by workloads.py, no dataset)",
        "config": {"workload": w.description, "tokens": T, "segments": w.tree.num_segments,
                   "q_heads": w.hq, "kv_heads": w.hkv, "head_dim": D, "useful_pairs_per_head": pairs,
                   "tile_tokens": 128 // G, "parallelism": f"replicas x{ws}" if ws > 1 else "1 GPU",
                   "l2": "inputs larger than L2 (%d MiB here; Q and dO %d MiB each); no flush between steps"
                         % (l2_bytes >> 20, q.numel() * 2 >> 20)},
        "tokens_per_s": round(ws * T / (ms_step * 1e-3), 1),
        "tokens_per_s_fwd": round(ws * T / (med_fwd * 1e-3), 1),
        "tokens_per_s_bwd": round(ws * T / (med_bwd * 1e-3), 1),
        "tile_efficiency": tile_efficiency(spc, plan, G, pairs),
        "cold_l2": cold,
        "fwd": {"ms": round(med_fwd, 4), "useful_tflops": round(fwd_tflops, 2),
                "frac_of_peak": round(fwd_tflops / p_burst, 4) if p_burst else None},
        "bwd": {"ms": round(med_bwd, 4), "useful_tflops": round(bwd_tflops, 2),
                "frac_of_peak": round(bwd_tflops / p_burst, 4) if p_burst else None},
        "edge_gather": {"ms": round(statistics.median(gat_ms), 4),
                        "gbs": round(2 * gathered.numel() * 2 / (statistics.median(gat_ms) * 1e-3) / 1e9, 1)
                        if gathered is not None and statistics.median(gat_ms) > 0 else None,
                        "frac_of_hbm_peak": round(2 * gathered.numel() * 2 / (statistics.median(gat_ms) * 1e-3)
                                                  / 1e9 / p_hbm, 4)
                        if gathered is not None and statistics.median(gat_ms) > 0 and p_hbm else None},
        "frac_of_bf16_peak": round(value / ws / p_burst, 4) if p_burst else None,
        "plan_ms": round(plan_ms, 3),
        "roofline": {
            "kernel": "bwd_tc_kernel (the backward's main kernel), timed alone by events around its launch",
            "bound": "tensor", "achieved": round(f_bwd / (mean_main * 1e-3) / 1e12, 2),
            "peak": p_burst, "unit": "TFLOP/s",
            "frac": round(f_bwd / (mean_main * 1e-3) / 1e12 / p_burst, 4) if p_burst else None,
            "ms": round(mean_main, 4), "flops_per_launch": f_bwd,
            "traffic": traffic_bwd[0], "traffic_source": traffic_bwd[1], "traffic_kernel": "bwd_tc_kernel",
            "algorithmic_bytes": algo_bwd,
            "peak_source": f"bf16 burst, {src_burst} (the kernel runs {mean_main:.1f} ms at a time inside a "
                           f"{total_ms / 1e3:.2f} s timed region)",
            "frac_of_sustained_peak": round(f_bwd / (mean_main * 1e-3) / 1e12 / p_sust, 4) if p_sust else None,
            "sustained_peak": p_sust, "sustained_peak_source": f"bf16 sustained, {src_sust}",
            "whole_call": {"ms": round(mean_bwd, 4), "achieved": round(f_bwd / (mean_bwd * 1e-3) / 1e12, 2),
                           "frac": round(f_bwd / (mean_bwd * 1e-3) / 1e12 / p_burst, 4) if p_burst else None}},
        "roofline_fwd": {
            "kernel": "tree_attn_fwd", "bound": "tensor",
            "achieved": round(f_fwd / (mean_fwd * 1e-3) / 1e12, 2), "peak": p_burst, "unit": "TFLOP/s",
            "frac": round(f_fwd / (mean_fwd * 1e-3) / 1e12 / p_burst, 4) if p_burst else None,
            "traffic": traffic_fwd[0], "traffic_source": traffic_fwd[1], "traffic_kernel": "fwd_tc_kernel",
            "algorithmic_bytes": algo_fwd, "peak_source": f"bf16 burst, {src_burst}"},
        "gpu_launches": args.steps * sum(LAUNCHES_PER_STEP.values() if hidden is not None
                                         else [LAUNCHES_PER_STEP["fwd"], LAUNCHES_PER_STEP["bwd"]]),
        "clocks": clk,
        "e2e": e2e,
        "bwd_deterministic": det,
        "fwd_paired_sm": paired,
        "fragments": fragment_summary(spc, w, args.fragment_cap),
        "lm_head": lm_head,
    }
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        cb = run_oracle_sample(w, args.cpu_flops)
        line["cpu_baseline"] = {"value": round(cb["useful_flops"] / cb["times"][0] / 1e12, 6), "unit": UNIT,
                                "cores": cb["cores"], "kind": "oracle", "sample": cb["sample"],
                                "seconds": round(cb["times"][0], 2)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def fragment_summary(spc, w, cap: int):
    """Bounded fragments of the workload's tree (host planner): count and token duplication.  A cap
    below the tree's longest root path is infeasible; it is doubled until it holds that path."""
    need = 0
    depth_tokens = np.zeros(w.tree.num_segments, dtype=np.int64)
    for s in range(w.tree.num_segments):
        p = int(w.tree.parent[s])
        depth_tokens[s] = (depth_tokens[p] if p >= 0 else 0) + int(w.tree.seg_len[s])
        need = max(need, int(depth_tokens[s]))
    asked = cap
    while cap < need:
        cap *= 2
    t0 = time.perf_counter()
    try:
        f = spc.fragment_plan(w.tree, cap)
    except RuntimeError as e:
        return {"cap": cap, "error": str(e)}
    ms = (time.perf_counter() - t0) * 1e3
    return {"cap": cap, **({"cap_asked": asked, "longest_root_path": need} if cap != asked else {}),
            "fragments": f["num_fragments"], "physical_tokens": f["physical_tokens"],
            "fragment_tokens": f["fragment_tokens"],
            "duplication": round(f["fragment_tokens"] / max(1, f["physical_tokens"]), 4), "plan_ms": round(ms, 3)}


def run_deterministic_bwd(args, spc, plan, q, k, v, o, lse, do, dq, dk, dv, ws_buf, scale, status, dev, f_bwd,
                          p_burst):
    """The backward with dQ formed per query tile (no atomics), timed like the step's backward."""
    import torch
    stream = torch.cuda.current_stream(dev)
    ms, main = [], []
    for i in range(args.warmup + args.steps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        for x_ in e:
            x_.record(stream)
        e[0].record(stream)
        spc.sp_tree_attn_bwd_timed(plan, q, k, v, o, lse, do, dq, dk, dv, ws_buf, scale, True, e[1], e[2], status)
        e[3].record(stream)
        torch.cuda.synchronize(dev)
        if i >= args.warmup:
            ms.append(e[0].elapsed_time(e[3]))
            main.append(e[1].elapsed_time(e[2]))
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item()} in the deterministic backward")
    t = statistics.median(ms)
    tf = f_bwd / (t * 1e-3) / 1e12
    tm = statistics.median(main)
    return {"ms": round(t, 4), "useful_tflops": round(tf, 2), "frac_of_peak": round(tf / p_burst, 4) if p_burst else None,
            "key_block_kernel_ms": round(tm, 4), "query_tile_kernel_and_preprocess_ms": round(t - tm, 4),
            "launches": 3}


def run_paired_fwd(args, spc, plan, q, k, v, o, lse, scale, status, dev, f_fwd, p_burst):
    """The forward on pairs of SMs (cta_group::2 products), timed like the step's forward; null where it
    does not apply (head_dim other than 128)."""
    import torch
    if q.shape[2] != 128:
        return None
    stream = torch.cuda.current_stream(dev)
    ms = []
    for i in range(args.warmup + args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        spc.sp_tree_attn_fwd_paired(plan, q, k, v, o, lse, scale, status)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if i >= args.warmup:
            ms.append(e0.elapsed_time(e1))
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item()} in the paired-SM forward")
    t = statistics.median(ms)
    tf = f_fwd / (t * 1e-3) / 1e12
    return {"ms": round(t, 4), "useful_tflops": round(tf, 2),
            "frac_of_peak": round(tf / p_burst, 4) if p_burst else None, "launches": 1}


def run_lm_head(args, spc, w, gathered, idx, dev, p_burst, p_sust):
    """The sampled-edge vocabulary head after the step: log-probabilities of the
    gathered states (forward) and their gradients, then the gradient's scatter
    back to the hidden states.  Timed separately from the attention step."""
    import torch
    E, Hd = gathered.shape
    x = W.draw_lm_head(E, Hd, args.lm_vocab, seed=w.seed)
    V = x["weight"].shape[0]
    wt, y, g = x["weight"].to(dev), x["labels"].to(dev), x["grad_logprob"].to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    lp = torch.empty(E, dtype=torch.float32, device=dev)
    lse = torch.empty(E, dtype=torch.float32, device=dev)
    dh = torch.empty((E, Hd), dtype=torch.float32, device=dev)
    dw = torch.empty((V, Hd), dtype=torch.float32, device=dev)
    ghid = torch.empty((w.T, Hd), dtype=torch.float32, device=dev)
    ws_f = torch.empty(spc.sp_edge_logprob_workspace_bytes(E, V), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(spc.sp_edge_logprob_bwd_workspace_bytes(E, V), dtype=torch.uint8, device=dev)
    ws_g = torch.empty(max(256, spc.sp_edge_gather_bwd_workspace_bytes(w.T, E)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    times = {"fwd": [], "bwd": [], "gather_bwd": []}
    for i in range(args.warmup + args.steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ev[0].record(stream)
        spc.sp_edge_logprob(gathered, wt, y, lp, lse, ws_f, st)
        ev[1].record(stream)
        spc.sp_edge_logprob_bwd(gathered, wt, y, lse, g, dh, dw, ws_b, st)
        ev[2].record(stream)
        spc.sp_edge_gather_bwd(dh, idx, ghid, ws_g, st)
        ev[3].record(stream)
        torch.cuda.synchronize(dev)
        if i >= args.warmup:
            times["fwd"].append(ev[0].elapsed_time(ev[1]))
            times["bwd"].append(ev[1].elapsed_time(ev[2]))
            times["gather_bwd"].append(ev[2].elapsed_time(ev[3]))
    if st.item() != 0:
        raise RuntimeError(f"device status {st.item()} in the vocabulary head")
    f = 2.0 * E * Hd * V
    t_f, t_b = statistics.median(times["fwd"]), statistics.median(times["bwd"])
    return {"actions": E, "hidden": Hd, "vocab": V, "dtype": "bf16 in, fp32 accumulate",
            "fwd": {"ms": round(t_f, 4), "tflops": round(f / t_f / 1e9, 1),
                    "frac_of_peak": round(f / t_f / 1e9 / p_burst, 4) if p_burst else None},
            "bwd": {"ms": round(t_b, 4), "tflops": round(3 * f / t_b / 1e9, 1),
                    "frac_of_peak": round(3 * f / t_b / 1e9 / p_sust, 4) if p_sust else None},
            "gather_bwd_ms": round(statistics.median(times["gather_bwd"]), 4),
            "flops": {"fwd": f, "bwd": 3 * f}, "launches_per_step": {"fwd": 2, "bwd": 3, "gather_bwd": 5}}


def run_e2e(args, spc, w, x, dev, flops_per_step):
    """Same metric through the public API from pinned host buffers.  Every step
    plans the tree and uploads the plan, copies that step's inputs in, runs
    forward, backward and the gather, and copies dQ, dK, dV and the gathered
    rows out.  Steps are pipelined the way a training loop would run them: three
    device buffer sets, inputs copied on one stream and results on another
    while the previous steps compute (the copies of a step still precede and
    follow its own compute).  A step's inputs start copying in as soon as the
    step three back has computed, so a copy that runs late (the host-device link
    is shared by both directions) still has two steps of compute to hide behind."""
    import torch
    G = w.hq // w.hkv
    host = {n: t.pin_memory() for n, t in x.items()}
    idx_h = torch.from_numpy(w.edge_idx).pin_memory() if w.edge_idx is not None else None
    nbuf = 3
    sets = []
    for _ in range(nbuf):
        d = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
        d["idx"] = torch.empty_like(idx_h, device=dev) if idx_h is not None else None
        d["ws"] = spc.bwd_workspace(d["q"])
        d["o"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty((w.hq, w.T), dtype=torch.float32, device=dev)
        d["dq"], d["dk"], d["dv"] = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])
        d["g"] = torch.empty((idx_h.shape[0], host["hidden"].shape[1]), dtype=torch.bfloat16, device=dev) \
            if idx_h is not None and "hidden" in host else None
        d["out_h"] = {n: torch.empty_like(d[n], device="cpu").pin_memory() for n in ("dq", "dk", "dv")}
        d["g_h"] = torch.empty_like(d["g"], device="cpu").pin_memory() if d["g"] is not None else None
        sets.append(d)
    h2d = sum(t.numel() * t.element_size() for t in host.values()) + \
        (idx_h.numel() * 4 if idx_h is not None else 0)
    d2h = sum(t.numel() * t.element_size() for t in sets[0]["out_h"].values()) + \
        (sets[0]["g_h"].numel() * 2 if sets[0]["g_h"] is not None else 0)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    comp = torch.cuda.current_stream(dev)
    s_plan = torch.cuda.Stream(device=dev)
    # copies in on three streams and out on two, so several copy engines share the link: the tensors of
    # each direction are dealt to the streams largest first, each to the stream with the fewest bytes so far
    s_in = [torch.cuda.Stream(device=dev) for _ in range(3)]
    s_out = [torch.cuda.Stream(device=dev) for _ in range(2)]

    def deal(names, nbytes, k):
        lanes, load = [[] for _ in range(k)], [0] * k
        for n in sorted(names, key=lambda n_: -nbytes[n_]):
            i = load.index(min(load))
            lanes[i].append(n)
            load[i] += nbytes[n]
        return lanes
    in_bytes = {n: t.numel() * t.element_size() for n, t in host.items()}
    if idx_h is not None:
        in_bytes["idx"] = idx_h.numel() * idx_h.element_size()
    # the forward's inputs first, so a step's forward starts while the rest is still coming in
    first = [n for n in ("q", "k", "v") if n in in_bytes]
    in_lanes = [deal(first, in_bytes, len(s_in)), deal([n for n in in_bytes if n not in first], in_bytes, len(s_in))]
    plan_buf = [None] * nbuf  # per buffer set: the device buffer its steps' plans are uploaded into
    ev_comp = [torch.cuda.Event() for _ in range(nbuf)]   # compute of the set's last step done
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]    # results of the set's last step copied out
    for b in range(nbuf):
        ev_comp[b].record(comp)
        ev_out[b].record(comp)
    plans = []
    marks = []  # per step: events on the streams and host times (the breakdown of the end-to-end time)

    def ev():
        e = torch.cuda.Event(enable_timing=True)
        return e

    def step(i):
        d = sets[i % nbuf]
        b = i % nbuf
        m = {"host_t0": time.perf_counter()}
        plan = spc.tree_plan(w.tree, 128 // G, 128, 0, upload=False)
        m["host_plan_ms"] = (time.perf_counter() - m["host_t0"]) * 1e3
        need = spc.sp_plan_device_bytes(plan)
        if plan_buf[b] is None or plan_buf[b].numel() < need:
            plan_buf[b] = torch.empty(2 * need, dtype=torch.uint8, device=dev)
        # the set's buffer is free once its previous step (three back) has computed; the upload goes on an
        # idle stream of its own (a copy from pageable host memory queued behind busy work would stall)
        t_wait = time.perf_counter()
        ev_comp[b].synchronize()
        m["host_wait_ms"] = (time.perf_counter() - t_wait) * 1e3
        t_up = time.perf_counter()
        m["upload0"], m["upload1"] = ev(), ev()
        m["upload0"].record(s_plan)
        spc.sp_plan_upload_to(plan, plan_buf[b], s_plan)
        m["upload1"].record(s_plan)
        m["host_upload_ms"] = (time.perf_counter() - t_up) * 1e3
        comp.wait_event(m["upload1"])
        plans.append(plan)
        m["h2d0"], m["h2d_fwd"], m["h2d1"] = ev(), ev(), ev()
        s_in[0].wait_event(ev_comp[b])  # the set's inputs are free once its previous step has computed
        m["h2d0"].record(s_in[0])
        for si in s_in[1:]:
            si.wait_event(m["h2d0"])
        for phase, lanes in enumerate(in_lanes):
            for si, lane_names in zip(s_in, lanes):
                if phase == 1:
                    si.wait_event(m["h2d_fwd"])  # the forward's inputs get the whole link first
                with torch.cuda.stream(si):
                    for n in lane_names:
                        d[n].copy_(idx_h if n == "idx" else host[n], non_blocking=True)
            for si in s_in[1:]:
                e_ = torch.cuda.Event()
                e_.record(si)
                s_in[0].wait_event(e_)
            m["h2d_fwd" if phase == 0 else "h2d1"].record(s_in[0])
        comp.wait_event(m["h2d_fwd"])  # Q, K, V in: the forward may start
        m["comp0"], m["comp1"] = ev(), ev()
        m["comp0"].record(comp)
        spc.sp_tree_attn_fwd(plan, d["q"], d["k"], d["v"], d["o"], d["lse"], w.softmax_scale, status)
        comp.wait_event(m["h2d1"])  # dO, the hidden rows and the edge indices in
        comp.wait_event(ev_out[b])  # the set's result buffers have been copied out
        spc.sp_tree_attn_bwd(plan, d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], d["dq"], d["dk"], d["dv"],
                             d["ws"], w.softmax_scale, status)
        if d["g"] is not None:
            spc.sp_edge_gather(d["hidden"], d["idx"], d["g"], status)
        m["comp1"].record(comp)
        ev_comp[b].record(comp)
        m["d2h0"], m["d2h1"] = ev(), ev()
        s_out[0].wait_event(ev_comp[b])
        m["d2h0"].record(s_out[0])
        outs = [(d["out_h"][n], d[n]) for n in ("dq", "dk", "dv")] + \
            ([(d["g_h"], d["g"])] if d["g"] is not None else [])
        out_bytes = {i: src.numel() * src.element_size() for i, (_, src) in enumerate(outs)}
        for so, lane_ids in zip(s_out, deal(list(out_bytes), out_bytes, len(s_out))):
            so.wait_event(m["d2h0"])
            with torch.cuda.stream(so):
                for i in lane_ids:
                    outs[i][0].copy_(outs[i][1], non_blocking=True)
        for so in s_out[1:]:
            e_ = torch.cuda.Event()
            e_.record(so)
            s_out[0].wait_event(e_)
        m["d2h1"].record(s_out[0])
        ev_out[b].record(s_out[0])
        m["host_ms"] = (time.perf_counter() - m["host_t0"]) * 1e3
        marks.append(m)

    for i in range(max(1, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    n = max(2, min(args.steps, 20))
    marks.clear()
    t_start = ev()
    t_start.record(comp)
    t0 = time.perf_counter()
    for i in range(n):
        step(i)
    torch.cuda.synchronize(dev)
    el = (time.perf_counter() - t0) / n
    breakdown = e2e_breakdown(marks, t_start, el * 1e3)
    for p_ in plans:
        p_.close()
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item()} in the end-to-end run")
    return {"value": round(flops_per_step / el / 1e12, 3), "unit": UNIT, "ms_per_step": round(el * 1e3, 3),
            "steps": n, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipelined": "3 buffer sets; inputs in on three streams (Q, K, V first: a step's forward starts before "
                         "dO and the hidden rows are in), results out on two, the next steps' copies overlapping "
                         "this step's compute; each step's plan uploaded into a reused device buffer",
            "includes": "tree_plan + plan upload + H2D of q,k,v,dO,hidden,idx + fwd + bwd + edge_gather + "
                        "D2H of dQ,dK,dV and gathered rows",
            "breakdown": breakdown}


def e2e_breakdown(marks, t_start, step_ms):
    """Where the end-to-end time per step goes, from the events of the timed steps (ms, medians over steps
    unless said): compute, the copies in and out, the plan upload and host times; the compute stream's idle
    time between steps; and the pipeline's fill (before the first compute) and drain (after the last)."""
    med = lambda xs: round(statistics.median(xs), 4) if xs else None  # noqa: E731
    el = lambda a, b: a.elapsed_time(b)  # noqa: E731
    comp = [el(m["comp0"], m["comp1"]) for m in marks]
    gaps = [el(marks[i]["comp1"], marks[i + 1]["comp0"]) for i in range(len(marks) - 1)]
    total = el(t_start, marks[-1]["d2h1"])
    fill = el(t_start, marks[0]["comp0"])
    drain = el(marks[-1]["comp1"], marks[-1]["d2h1"])
    return {"compute_ms": med(comp), "h2d_ms": med([el(m["h2d0"], m["h2d1"]) for m in marks]),
            "h2d_forward_inputs_ms": med([el(m["h2d0"], m["h2d_fwd"]) for m in marks if "h2d_fwd" in m]),
            "d2h_ms": med([el(m["d2h0"], m["d2h1"]) for m in marks]),
            "upload_ms": med([el(m["upload0"], m["upload1"]) for m in marks]),
            "compute_idle_between_steps_ms": med(gaps), "compute_idle_total_ms": round(sum(gaps), 4),
            "compute_idle_max_ms": round(max(gaps), 4) if gaps else None,
            "compute_gaps_ms": [round(x, 3) for x in gaps],
            "h2d_max_ms": round(max(el(m["h2d0"], m["h2d1"]) for m in marks), 4),
            "fill_ms": round(fill, 4), "drain_ms": round(drain, 4), "steps": len(marks),
            "device_span_ms": round(total, 4), "step_ms_host_clock": round(step_ms, 4),
            "host_plan_ms": med([m["host_plan_ms"] for m in marks]),
            "host_upload_ms": med([m["host_upload_ms"] for m in marks]),
            "host_upload_max_ms": round(max(m["host_upload_ms"] for m in marks), 4),
            "host_wait_max_ms": round(max(m["host_wait_ms"] for m in marks), 4),
            "h2d_ms_by_step": [round(el(m["h2d0"], m["h2d1"]), 2) for m in marks],
            "host_wait_ms": med([m["host_wait_ms"] for m in marks]),
            "host_step_ms": med([m["host_ms"] for m in marks])}


def cta_tail_stats(rec):
    """Tail of one launch from its per-CTA records [n, 4] = (start ns, end ns, SM, 0): the launch's span,
    the share of SM-time left idle after each SM's last CTA ended (the last wave's idle time), and the
    share of SM-time the CTAs occupied."""
    rec = rec[rec[:, 1] > 0]
    start, end, sm = rec[:, 0].astype(np.float64), rec[:, 1].astype(np.float64), rec[:, 2]
    t0, t1 = start.min(), end.max()
    span = t1 - t0
    sms = np.unique(sm)
    last = np.array([end[sm == x].max() for x in sms])
    busy = float((end - start).sum() / (span * len(sms)))
    dur = end - start
    return {"ctas": int(len(rec)), "sms": int(len(sms)), "span_us": round(span / 1e3, 2),
            "tail_idle_frac": round(float((t1 - last).sum() / (span * len(sms))), 4),
            "busy_frac": round(busy, 4), "longest_cta_us": round(float(dur.max()) / 1e3, 2),
            "median_cta_us": round(float(np.median(dur)) / 1e3, 2),
            "last_sm_idle_us": round(float(t1 - last.min()) / 1e3, 2)}


def run_cta_tail(args):
    """Per-CTA start/end times of the tensor-core kernels (sp_debug_cta_clock) on one workload: how much
    SM-time each launch leaves idle at its end, the figure split-KV work division would recover."""
    import torch
    dev = torch.device("cuda", 0)
    import shared_prefix_causal_gb300 as spc
    w = W.get(args.config)
    G = w.hq // w.hkv
    x = W.draw_tensors(w, "bf16")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    plan = spc.tree_plan(w.tree, 128 // G, 128, 0)
    o = torch.empty_like(q)
    lse = torch.empty((w.hq, w.T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = spc.bwd_workspace(q)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    buf = torch.zeros((1 << 20, 4), dtype=torch.int64, device=dev)
    scale = w.softmax_scale
    calls = {
        "forward": (spc.CLOCK_FORWARD, lambda: spc.sp_tree_attn_fwd(plan, q, k, v, o, lse, scale, st)),
        "backward key blocks (default)": (spc.CLOCK_KEY_BLOCKS, lambda: spc.sp_tree_attn_bwd(
            plan, q, k, v, o, lse, do, dq, dk, dv, ws, scale, st)),
        "backward key blocks (deterministic)": (spc.CLOCK_KEY_BLOCKS, lambda: spc.sp_tree_attn_bwd_deterministic(
            plan, q, k, v, o, lse, do, dq, dk, dv, ws, scale, st)),
        "backward query tiles (deterministic dQ)": (spc.CLOCK_QUERY_TILES, lambda: spc.sp_tree_attn_bwd_deterministic(
            plan, q, k, v, o, lse, do, dq, dk, dv, ws, scale, st)),
    }
    out = {"workload": w.description, "tokens": w.T, "kernels": {}}
    for name, (kid, fn) in calls.items():
        for _ in range(2):  # warm-up
            fn()
        buf.zero_()
        spc.sp_debug_cta_clock(kid, buf)
        fn()
        torch.cuda.synchronize(dev)
        spc.sp_debug_cta_clock(0)
        if st.item() != 0:
            raise RuntimeError(f"device status {st.item()} in {name}")
        out["kernels"][name] = cta_tail_stats(buf.cpu().numpy())
    print(json.dumps(out), flush=True)


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    w = W.get(args.config)
    reps = args.warmup + args.steps
    # the whole run stays within its budget: with many steps each step's sample shrinks
    r = run_oracle_sample(w, min(args.ref_flops, args.ref_total_flops / max(1, reps)), reps=reps)
    times = r["times"][args.warmup:]
    total = sum(times)
    value = r["useful_flops"] * len(times) / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / len(times) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; inputs drawn by workloads.py, no dataset)",
        "config": {"workload": w.description, "sample_tokens_per_step": r["tokens"]},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                         "sample": r["sample"]},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="agent", choices=list(W.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--no-lm-head", action="store_true", help="skip the vocabulary-head measurement")
    ap.add_argument("--lm-vocab", type=int, default=W.LM_HEAD_VOCAB, help="vocabulary size of the vocabulary head")
    ap.add_argument("--fragment-cap", type=int, default=32768, help="token cap of the bounded-fragment summary")
    ap.add_argument("--cpu-flops", type=float, default=6e11, help="fp64 flop budget of the CPU-baseline sample")
    ap.add_argument("--ref-flops", type=float, default=1.2e11, help="fp64 flop budget per reference step")
    ap.add_argument("--ref-total-flops", type=float, default=4e12,
                    help="fp64 flop budget of the whole reference run (warm-up and timed steps together)")
    ap.add_argument("--cta-tail", action="store_true",
                    help="instead of the bench line: per-CTA timing of the tensor-core kernels (launch tails)")
    ap.add_argument("--_oracle-child", dest="oracle_child", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_child:
        oracle_child(json.loads(args.oracle_child))
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.cta_tail:
        run_cta_tail(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
