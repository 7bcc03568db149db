"""Static rules for the CUDA sources, checked on the CPU.

The GPU is shared with other users, so a kernel must never hang or trap it.
These rules keep later edits from quietly breaking that:
  * every mbarrier poll (CTA or cluster scope) goes through the bounded waits
    of ``pipeline.cuh``;
  * no loop without a condition outside those waits;
  * no trap, breakpoint or device assert;
  * every TMEM allocation (one SM or a pair) is matched by a deallocation that
    no early return skips (returns inside a lambda leave only the lambda).
The sources are read as text with comments removed; nothing is compiled.
"""
import glob
import os
import re

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "shared_prefix_causal_gb300",
                    "csrc")
DEVICE_FILES = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")))


def _code(path):
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", lambda m: "\n" * m.group(0).count("\n"), text, flags=re.S)
    return re.sub(r"//[^\n]*", "", text)


def _name(path):
    return os.path.basename(path)


def _lambda_spans(code):
    """(start, end) character spans of lambda bodies ``[...](...) ... { ... }``."""
    spans = []
    for m in re.finditer(r"\[[&=]?[\w, &]*\]\s*\([^)]*\)[^{;]*\{", code):
        depth, i = 1, m.end()
        while depth and i < len(code):
            depth += {"{": 1, "}": -1}.get(code[i], 0)
            i += 1
        spans.append((m.end(), i))
    return spans


def test_device_sources_exist():
    names = {_name(p) for p in DEVICE_FILES}
    assert {"attn_fwd_sm103a.cu", "attn_bwd_sm103a.cu", "pipeline.cuh", "sm103_ptx.cuh"} <= names


@pytest.mark.parametrize("path", DEVICE_FILES, ids=_name)
def test_mbarrier_polls_only_in_the_bounded_waits(path):
    calls = re.findall(r"\bmbar_try_wait(?:_cluster)?\s*\(", _code(path))
    if _name(path) == "sm103_ptx.cuh":
        assert len(calls) == 2  # the definitions (CTA and cluster scope)
    elif _name(path) != "pipeline.cuh":
        assert not calls, "poll an mbarrier through spc::Ctl (bounded), not directly"


@pytest.mark.parametrize("path", DEVICE_FILES, ids=_name)
def test_no_trap_breakpoint_or_device_assert(path):
    code = _code(path)
    for pat in (r"__trap\s*\(", r"\btrap\s*;", r"\bbrkpt\b", r"\bassert\s*\(", r"__brkpt\s*\("):
        assert not re.search(pat, code), f"{_name(path)}: {pat}"


@pytest.mark.parametrize("path", DEVICE_FILES, ids=_name)
def test_loops_without_a_condition_only_in_the_bounded_waits(path):
    code = _code(path)
    endless = re.findall(r"\bfor\s*\([^;()]*;\s*;[^)]*\)|\bwhile\s*\(\s*(?:1|true)\s*\)", code)
    if _name(path) == "pipeline.cuh":
        assert len(endless) == 1  # Ctl::wait, which counts its polls against the limit
    else:
        assert not endless, f"{_name(path)}: {endless}"


@pytest.mark.parametrize("path", DEVICE_FILES, ids=_name)
def test_tmem_is_freed_on_every_path(path):
    code = _code(path)
    allocs = [m.start() for m in re.finditer(r"\btmem_alloc(?:_pair)?\s*\(", code)]
    deallocs = [m.start() for m in re.finditer(r"\btmem_dealloc(?:_pair)?\s*\(", code)]
    if _name(path) == "sm103_ptx.cuh":
        return  # the helpers' definitions
    assert len(allocs) == len(deallocs)
    spans = _lambda_spans(code)
    for a, d in zip(allocs, deallocs):
        assert a < d
        for m in re.finditer(r"\breturn\b", code[a:d]):
            pos = a + m.start()
            assert any(s <= pos < e for s, e in spans), \
                f"{_name(path)}: a return at line {code[:pos].count(chr(10)) + 1} skips the TMEM deallocation"


def test_the_rules_catch_planted_violations(tmp_path):
    """The checks above, applied to a source with one violation of each kind, all fire."""
    bad = tmp_path / "bad.cu"
    bad.write_text(
        "__global__ void k(){ tmem_alloc(0, 32);\n"
        "  if (threadIdx.x) return;\n"
        "  while (true) { if (mbar_try_wait(0, 0)) break; }\n"
        "  __trap();\n"
        "  tmem_dealloc(0, 32); }\n")
    p = str(bad)
    for check in (test_mbarrier_polls_only_in_the_bounded_waits, test_no_trap_breakpoint_or_device_assert,
                  test_loops_without_a_condition_only_in_the_bounded_waits, test_tmem_is_freed_on_every_path):
        with pytest.raises(AssertionError):
            check(p)
    ok = tmp_path / "ok.cu"
    ok.write_text("__global__ void k(){ tmem_alloc(0, 32);\n"
                  "  auto f = [&](int m) -> bool { if (m) return false; return true; };\n"
                  "  f(1); tmem_dealloc(0, 32); }\n")
    test_tmem_is_freed_on_every_path(str(ok))
