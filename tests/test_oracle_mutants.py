"""The oracle's pins catch planted mistakes.

Each case below plants one plausible mistake in a private copy of the oracle
package: a dropped term, a wrong sign or bound, a wrong index or a transposed
operand.  The case then runs the pins of ``test_oracle.py`` against that copy
and expects at least one of them to fail.  A mistake that every pin tolerates
would be a mistake the oracle could carry into every parity test unnoticed.

Everything runs on the CPU against the copy; the real ``oracle`` package and
the CUDA library are untouched.
"""
import contextlib
import importlib.util
import shutil
import sys
from pathlib import Path

import pytest

import oracle
import test_oracle as P

ORACLE_DIR = Path(__file__).resolve().parent.parent / "oracle"
MUTANT_PKG = "_oracle_mutant"

# (module, text in the oracle, replacement, what the mistake is)
MUTANTS = [
    # tree: validation, ancestry, brute-force visibility
    ("tree", "if seg_len[s] < 1:", "if seg_len[s] < 0:", "empty segments accepted"),
    ("tree", "want = 0 if p == -1 else depth[p] + 1", "want = 0 if p == -1 else depth[p]",
     "depth not incremented"),
    ("tree", "                a = parent[a]\n            if p not in on_path",
     "                a = -1\n            if p not in on_path", "preorder check sees only the previous segment"),
    ("tree", "if seg_start[s] != pos:", "if seg_start[s] < pos:", "gaps between segments accepted"),
    ("tree", "    return out[::-1]\n", "    return out\n", "ancestors leaf first"),
    ("tree", "segs = ancestors(parent, leaf) + [leaf]", "segs = ancestors(parent, leaf)",
     "root-to-leaf path drops the leaf"),
    ("tree", "todo.extend(ch[a])", "todo.extend(ch[a][:1])", "descendants follow the first child only"),
    ("tree", "m[i, j] = j <= i", "m[i, j] = j < i", "diagonal not visible"),
    ("tree", "m[i, j] = int(seg[j]) in anc", "m[i, j] = j <= i", "plain causal instead of the tree rule"),
    ("tree", "        if p >= 0:\n            ch[int(p)].append(s)",
     "        if p > 0:\n            ch[int(p)].append(s)", "children of segment 0 lost"),
    # plan: tiles, ranges, order, backward table
    ("plan", "if out and out[-1][1] == a:", "if False:", "touching ranges not merged"),
    ("plan", "q1 = min(q0 + tile_tokens, a1)", "q1 = q0 + tile_tokens", "tiles cross the segment end"),
    ("plan", "rng = _merge(anc_iv + [(a0, q1)])", "rng = _merge(anc_iv + [(a0, a1)])",
     "own range runs to the segment end"),
    ("plan", "key = (_root_of(parent, s), int(parent[s]), k, s)",
     "key = (_root_of(parent, s), int(parent[s]), s, k)", "siblings not interleaved by tile index"),
    ("plan", "key = (-sum(b - a for a, b in rng), s, k)", "key = (sum(b - a for a, b in rng), s, k)",
     "longest-first order reversed"),
    ("plan", "bwd.append((s, k0, min(k0 + kv_block, a1), k0, qe))",
     "bwd.append((s, k0, min(k0 + kv_block, a1), a0, qe))", "block queries start at the segment start"),
    ("plan", "bwd.sort(key=lambda r: (-(r[4] - r[3]), r[1]))", "bwd.sort(key=lambda r: (r[4] - r[3], r[1]))",
     "backward table ascending"),
    ("plan", "return max(int(seg_start[d]) + int(seg_len[d]) for d",
     "return max(int(seg_start[d]) for d", "subtree end is a start"),
    ("plan", "if r < rb + rc - 1 or j <= i:", "if r < rb + rc - 1 or j < i:",
     "forward mask expansion drops the diagonal"),
    ("plan", "                if j <= i:\n                    m[i, j] = True\n    return m",
     "                if j < i:\n                    m[i, j] = True\n    return m",
     "backward mask expansion drops the diagonal"),
    ("plan", "    while int(parent[s]) != -1:\n        s = int(parent[s])\n    return s",
     "    return int(parent[s])", "root of a segment is its parent"),
    # attention: unrolled paths, softmax, gradients, dense route
    ("attention", "S[np.arange(kmax)[None, :] > r[:, None]] = -np.inf",
     "S[np.arange(kmax)[None, :] >= r[:, None]] = -np.inf", "causal mask hides the diagonal"),
    ("attention", "LSE[c0:c0 + len(r)] = m + np.log(l)", "LSE[c0:c0 + len(r)] = np.log(l)",
     "LSE without the row maximum"),
    ("attention", "dS = P * (dP - Dv[:, None])\n            dQ[c0",
     "dS = P * dP\n            dQ[c0", "backward drops the rowsum(dO*O) term"),
    ("attention", "dQ[c0:c0 + len(r)] = scale * (dS @ kp[:kmax])", "dQ[c0:c0 + len(r)] = dS @ kp[:kmax]",
     "dQ without the softmax scale"),
    ("attention", "dK[:kmax] += scale * (dS.T @ qp[r])", "dK[:kmax] -= scale * (dS.T @ qp[r])",
     "dK with the wrong sign"),
    ("attention", "dV[:kmax] += P.T @ dOc", "dV[:kmax] += P.T @ Oc", "dV from O instead of dO"),
    ("attention", "Dv = (dOc * Oc).sum(axis=1)", "Dv = (dOc * Oc).sum(axis=1) * scale",
     "rowsum(dO*O) scaled"),
    ("attention", "h = group * G + j", "h = j * hkv + group", "query heads interleaved across KV heads"),
    ("attention", "own = np.nonzero(~seen[idx])[0]", "own = np.arange(len(idx))",
     "every copy of a prefix token owns its dO"),
    ("attention", "np.add.at(dK[:, g], idx, r[\"dK\"])", "dK[idx, g] = r[\"dK\"]",
     "prefix dK overwritten instead of summed over branches"),
    ("attention", "np.add.at(dV[:, g], idx, r[\"dV\"])", "dV[idx, g] = r[\"dV\"]",
     "prefix dV overwritten instead of summed over branches"),
    ("attention", "S = np.where(mask, S, -np.inf)", "S = np.where(mask.T, S, -np.inf)",
     "dense route reads the mask transposed"),
    ("attention", "dK[:, g] += scale * (dS.T @ q[:, h])", "dK[:, g] = scale * (dS.T @ q[:, h])",
     "dense dK keeps only the last query head of a group"),
    ("attention", "if int(idx[p]) not in seen", "if True", "subtree key gradients count shared rows twice"),
    ("attention", "kmax = int(r[-1]) + 1", "kmax = int(r[-1])", "last visible key cut off"),
    ("attention", "m = S.max(axis=1)\n        P = np.exp(S - m[:, None])", "m = S.max(axis=1) * 0\n        P = np.exp(S - m[:, None])",
     "softmax without the max shift (overflows on large scores)"),
    ("attention", "m = S.max(axis=1)\n        E = np.exp(S - m[:, None])", "m = S.max(axis=1) * 0\n        E = np.exp(S - m[:, None])",
     "dense softmax without the max shift"),
    ("attention", "O[:, h] = P[h] @ v[:, h // G]", "O[:, h] = P[h] @ v[:, h % k.shape[1]]", "dense route maps heads modulo"),
    ("attention", "LSE[hs, idx[new]] = r[\"LSE\"][:, new]", "LSE[hs, idx[new]] = r[\"LSE\"][::-1][:, new]",
     "LSE rows of a group's heads swapped"),
    ("attention", "dQ[idx[own], hs] += r[\"dQ\"]", "dQ[idx[own], hs] += r[\"dQ\"][:, ::-1]", "dQ heads of a group swapped"),
    ("attention", "dV[:, g] += P[h].T @ do[:, h]", "dV[:, g] += P[h] @ do[:, h]", "dense dV with P untransposed"),
    ("plan", "raw.sort(key=lambda r: r[0])", "raw.sort(key=lambda r: r[0], reverse=True)", "tile order reversed"),
    ("plan", "tiles.append((s, q0, q1, len(ranges), len(rng)))", "tiles.append((s, q0, q1, len(ranges), len(rng) - 1))",
     "range count drops the causal range"),
    ("gather", "return hidden[idx]", "return hidden[np.sort(idx)]", "gather rows sorted by source"),
    # gather
    ("gather", "if idx.size and (idx.min() < 0 or idx.max() >= T):", "if idx.size and (idx.min() < -1 or idx.max() >= T):",
     "gather accepts index -1 (NumPy would read the last row)"),
    ("gather", "if idx.size and (idx.min() < 0 or idx.max() >= num_tokens):",
     "if idx.size and (idx.min() < -1 or idx.max() >= num_tokens):", "gather backward accepts index -1"),
    ("gather", "out[idx[e]] += grad_out[e]", "out[idx[e]] = grad_out[e]",
     "gather backward keeps one of several duplicate rows"),
    # vocabulary head
    ("lm_head", "return m + np.log(np.exp(z - m[:, None]).sum(axis=1))",
     "return np.log(np.exp(z - m[:, None]).sum(axis=1))", "log-sum-exp without the row maximum"),
    ("lm_head", "return z[np.arange(len(labels)), labels] - lse, lse",
     "return z[np.arange(len(labels)), labels] + lse, lse", "log-probability adds the normaliser"),
    ("lm_head", "dz[np.arange(E), labels] += 1.0", "pass", "backward drops the label indicator"),
    ("lm_head", "    dz *= g[:, None]\n    return dz @ weight", "    return dz @ weight",
     "backward ignores the upstream gradient"),
    ("lm_head", "lse = log_sum_exp_rows(z)\n    dz = -np.exp(z[:, rows]",
     "lse = log_sum_exp_rows(z[:, rows])\n    dz = -np.exp(z[:, rows]", "row gradient normalised over the requested rows"),
    ("lm_head", "labels.min() < 0", "labels.min() < -1", "label -1 accepted (NumPy would read the last logit)"),
    # fragments
    ("fragments", "if cur and cur_tokens + extra > max_tokens:", "if cur and cur_tokens + extra >= max_tokens:",
     "a fragment never fills the cap exactly"),
    ("fragments", "cur.append((a, a == s))", "cur.append((a, True))", "repeated ancestors owned again"),
    ("fragments", "missing, extra = path, path_tokens", "missing, extra = [s], seg_len[s]",
     "a new fragment starts without the root path"),
    ("fragments", "if path_tokens > max_tokens:", "if path_tokens >= max_tokens:",
     "a root path exactly at the cap refused"),
    ("fragments", "assert (owners == 1).all()", "assert (owners >= 1).all()", "checker allows two owners"),
    ("fragments", "sum(int(seg_len[a]) for f in frags for a, _ in f)",
     "sum(int(seg_len[a]) for f in frags for a, o in f if o)", "physical tokens count owned segments only"),
    ("fragments", "assert int(parent[a]) in present", "assert int(parent[a]) >= -1",
     "checker does not check ancestor closure"),
]


# Not planted, because they cannot change any result (equivalent mistakes):
# descendants returned in stack order (only their maximum end and their set are
# used); fragment entries left unsorted, or root paths taken leaf first (a
# fragment's insertion order is already preorder: an ancestor missing from the
# current fragment precedes its first segment and so lies on that segment's root
# path); an index bound of T or a label bound of V (NumPy's own indexing raises
# there); a self-parent accepted by the parent check (the depth check refuses it).


def _cases(fn, limit=12):
    """The pin's parametrised calls (at most ``limit`` of them)."""
    marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
    if not marks:
        return [{}]
    (m,) = marks
    names = [s.strip() for s in m.args[0].split(",")]
    out = []
    for v in list(m.args[1])[:limit]:
        v = v if len(names) > 1 else (v,)
        out.append(dict(zip(names, v)))
    return out


# the finite-difference pin is by far the slowest: it runs last, once the cheaper pins have had their turn
PINS = [(name, kw) for name, fn in sorted(vars(P).items(), key=lambda kv: ("finite_differences" in kv[0], kv[0]))
        if name.startswith("test_") and callable(fn) for kw in _cases(fn)]


@contextlib.contextmanager
def _mutant(tmp_path, module, old, new):
    dst = tmp_path / MUTANT_PKG
    shutil.copytree(ORACLE_DIR, dst, ignore=shutil.ignore_patterns("__pycache__"))
    f = dst / f"{module}.py"
    text = f.read_text()
    assert text.count(old) == 1, f"{module}.py: the planted text must occur exactly once: {old!r}"
    f.write_text(text.replace(old, new))
    spec = importlib.util.spec_from_file_location(MUTANT_PKG, dst / "__init__.py",
                                                  submodule_search_locations=[str(dst)])
    pkg = importlib.util.module_from_spec(spec)
    sys.modules[MUTANT_PKG] = pkg
    try:
        spec.loader.exec_module(pkg)
        yield pkg
    finally:
        for k in [k for k in sys.modules if k == MUTANT_PKG or k.startswith(MUTANT_PKG + ".")]:
            del sys.modules[k]


def _install(monkeypatch, pkg):
    """Point the pins' module names (and in-function ``from oracle import ...``) at ``pkg``."""
    for alias, sub in (("A", "attention"), ("OG", "gather"), ("OP", "plan"), ("OT", "tree")):
        monkeypatch.setattr(P, alias, getattr(pkg, sub))
    for sub in ("tree", "plan", "attention", "gather", "lm_head", "fragments"):
        monkeypatch.setattr(oracle, sub, getattr(pkg, sub))


def _failing_pin(monkeypatch, pkg):
    """Name of the first pin that fails against ``pkg``, or None."""
    _install(monkeypatch, pkg)
    for name, kw in PINS:
        try:
            getattr(P, name)(**kw)
        except (Exception, pytest.fail.Exception) as e:  # an assertion, pytest.raises unmet, or an error
            return f"{name}{kw or ''}: {type(e).__name__}"
    return None


def test_unmutated_copy_passes_every_pin(tmp_path, monkeypatch):
    """The harness itself: an unchanged copy of the oracle passes the whole battery."""
    with _mutant(tmp_path, "tree", "def validate(", "def validate(") as pkg:
        assert _failing_pin(monkeypatch, pkg) is None


def test_every_oracle_module_is_mutated():
    mods = {p.stem for p in ORACLE_DIR.glob("*.py") if p.stem != "__init__"}
    assert mods == {m for m, *_ in MUTANTS}


@pytest.mark.filterwarnings("ignore::RuntimeWarning")  # a mutant may turn values into NaN
@pytest.mark.parametrize("module,old,new,what", MUTANTS, ids=[f"{m}: {w}" for m, _, _, w in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, monkeypatch, module, old, new, what):
    with _mutant(tmp_path, module, old, new) as pkg:
        caught = _failing_pin(monkeypatch, pkg)
    assert caught is not None, f"no pin fails when the oracle's {module} has this mistake: {what}"
