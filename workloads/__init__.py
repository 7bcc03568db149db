"""Seeded synthetic workloads for shared-prefix tree attention.

This module only *draws* inputs: tree shapes (segment lengths and parents in
DFS preorder), the Q/K/V/dO tensors, the hidden tensor and the sampled-edge
indices.  It holds none of the attention arithmetic, planning or masking, so
both the CUDA path and the CPU oracle can take their inputs from here without
sharing any of the method.

Tree layout (both pages describe it as DFS-linearized segments with
parent/depth metadata: issue #7386 "Describe the solution you'd like", and
PR #7387 "Summary"): segments are laid out in preorder; segment ``s`` owns
tokens ``[seg_start[s], seg_start[s] + seg_len[s])``; ``parent[s] < s`` or
``-1`` for a root; ``depth[s]`` is 0 for a root, else ``depth[parent] + 1``.

Drawing rules (fixed once, here):

* structure: ``numpy.random.default_rng(seed)``; an inclusive integer draw is
  ``rng.integers(lo, hi + 1)``, one call per value; a log-uniform length is
  ``int(exp(rng.uniform(ln lo, ln hi)))``.
* tensors: ``torch.Generator('cpu').manual_seed(seed)``; ``randn`` in fp32 in
  the order Q, K, V, dO, hidden, each drawn in chunks of ``CHUNK_TOKENS`` rows,
  then multiplied by the config's scale and rounded to bf16 (round to nearest
  even, which is what ``Tensor.to(torch.bfloat16)`` does).
* edge indices: drawn from the structure generator after the tree.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable

import numpy as np

CHUNK_TOKENS = 8192


@dataclasses.dataclass
class Tree:
    """DFS-preorder segment tree over a packed token buffer (int32 arrays)."""

    seg_start: np.ndarray
    seg_len: np.ndarray
    parent: np.ndarray
    depth: np.ndarray

    @property
    def num_segments(self) -> int:
        return int(self.seg_len.shape[0])

    @property
    def total_tokens(self) -> int:
        return int(self.seg_len.sum())


def tree_from_preorder(lengths, parents) -> Tree:
    """Build the int32 arrays from per-segment lengths and parents (preorder)."""
    seg_len = np.asarray(lengths, dtype=np.int32)
    parent = np.asarray(parents, dtype=np.int32)
    n = seg_len.shape[0]
    seg_start = np.zeros(n, dtype=np.int32)
    if n > 1:
        seg_start[1:] = np.cumsum(seg_len[:-1], dtype=np.int64).astype(np.int32)
    depth = np.zeros(n, dtype=np.int32)
    for s in range(n):
        p = int(parent[s])
        depth[s] = 0 if p < 0 else depth[p] + 1
    return Tree(seg_start, seg_len, parent, depth)


def _log_uniform(rng: np.random.Generator, lo: int, hi: int) -> int:
    return int(math.exp(rng.uniform(math.log(lo), math.log(hi))))


def _random_tree(rng, root_len_fn, child_len_fn, branch_lo, branch_hi, max_depth, cap):
    """Preorder recursive tree, cut at ``cap`` tokens (last segment truncated).

    Each visited node with depth < ``max_depth`` draws its number of children
    uniformly in ``[branch_lo, branch_hi]``, then the children are generated
    one after another, each drawing its own length when visited.  If the
    recursion finishes below ``cap`` tokens, the tree is discarded and a new
    one is drawn from the same (continuing) generator.
    """
    while True:
        lengths: list[int] = []
        parents: list[int] = []
        total = 0

        def visit(par: int, depth: int, length: int) -> bool:
            nonlocal total
            length = min(length, cap - total)
            me = len(lengths)
            lengths.append(length)
            parents.append(par)
            total += length
            if total >= cap:
                return True
            if depth < max_depth:
                nchild = int(rng.integers(branch_lo, branch_hi + 1))
                for _ in range(nchild):
                    if visit(me, depth + 1, child_len_fn()):
                        return True
            return False

        if visit(-1, 0, root_len_fn()):
            return tree_from_preorder(lengths, parents)


@dataclasses.dataclass
class Workload:
    name: str
    description: str
    tree: Tree
    hq: int
    hkv: int
    head_dim: int
    tensor_scale: float
    seed: int
    hidden_dim: int | None
    edge_idx: np.ndarray | None

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def T(self) -> int:
        return self.tree.total_tokens


def _leaf_tokens(tree: Tree) -> np.ndarray:
    has_child = np.zeros(tree.num_segments, dtype=bool)
    for p in tree.parent:
        if p >= 0:
            has_child[p] = True
    toks = [np.arange(tree.seg_start[s], tree.seg_start[s] + tree.seg_len[s])
            for s in range(tree.num_segments) if not has_child[s]]
    return np.concatenate(toks).astype(np.int32)


def tiny() -> Workload:
    """Root of 64 tokens; children 32, 48, 17; the 48-token child has
    grandchildren of 16 and 9 tokens (186 tokens); 2 q heads, 2 kv heads, D=64."""
    tree = tree_from_preorder([64, 32, 48, 16, 9, 17], [-1, 0, 0, 2, 2, 0])
    rng = np.random.default_rng(0)
    leaf = _leaf_tokens(tree)
    edge = rng.choice(leaf, size=8, replace=False).astype(np.int32)
    return Workload("tiny", "tiny tree 186 tokens, 2q/2kv heads, D=64", tree,
                    2, 2, 64, 1.0, 0, 256, edge)


def grpo_star() -> Workload:
    """One 2048-token prompt with 8 completions of U[256, 1024] tokens."""
    rng = np.random.default_rng(1)
    lens = [2048] + [int(rng.integers(256, 1024 + 1)) for _ in range(8)]
    tree = tree_from_preorder(lens, [-1] + [0] * 8)
    edge = np.arange(2048, tree.total_tokens, dtype=np.int32)
    return Workload("star", "GRPO star: prompt 2048 + 8 completions U[256,1024]; 32q/8kv, D=128",
                    tree, 32, 8, 128, 0.5, 1, 4096, edge)


def grpo_forest() -> Workload:
    """16 independent stars: prompt U[512, 4096], 16 completions U[128, 2048]."""
    rng = np.random.default_rng(2)
    lens: list[int] = []
    pars: list[int] = []
    for _ in range(16):
        root = len(lens)
        lens.append(int(rng.integers(512, 4096 + 1)))
        pars.append(-1)
        for _ in range(16):
            lens.append(int(rng.integers(128, 2048 + 1)))
            pars.append(root)
    tree = tree_from_preorder(lens, pars)
    return Workload("forest", "GRPO forest: 16 stars, prompts U[512,4096], 16 completions U[128,2048]; 32q/8kv, D=128",
                    tree, 32, 8, 128, 0.5, 2, None, None)


def agent_tree() -> Workload:
    """Random agent-call tree of 65,536 tokens: depth <= 8, 1-4 children per
    node, segment lengths log-uniform in [16, 4096]; 5% sampled-edge tokens."""
    rng = np.random.default_rng(3)
    tree = _random_tree(rng, lambda: _log_uniform(rng, 16, 4096), lambda: _log_uniform(rng, 16, 4096),
                        1, 4, 8, 65536)
    edge = np.nonzero(rng.random(tree.total_tokens) < 0.05)[0].astype(np.int32)
    return Workload("agent", "agent-call tree: 65536 tokens, depth<=8, branching U{1..4}, segments logU[16,4096]; 32q/8kv, D=128",
                    tree, 32, 8, 128, 0.5, 3, 4096, edge)


def long_fragment() -> Workload:
    """8K-token root trunk, then chains of depth <= 12 with 1-3 children per
    node and segments log-uniform in [64, 8192], capped at 131,072 tokens."""
    rng = np.random.default_rng(4)
    tree = _random_tree(rng, lambda: 8192, lambda: _log_uniform(rng, 64, 8192), 1, 3, 12, 131072)
    return Workload("long", "long bounded fragment: 131072 tokens, 8K trunk, depth<=12, branching U{1..3}, segments logU[64,8192]; 64q/8kv, D=128",
                    tree, 64, 8, 128, 0.5, 4, None, None)


# Reduced cases of the three large workloads, same recipes at a quarter to an
# eighth of the size: small enough for hardware-counter captures of a kernel,
# larger than L2 in their Q/K/V/dO, so their DRAM figures still mean something.

def grpo_forest_small() -> Workload:
    """2 independent stars of the forest recipe (prompt U[512, 4096], 16 completions U[128, 2048])."""
    rng = np.random.default_rng(2)
    lens: list[int] = []
    pars: list[int] = []
    for _ in range(2):
        root = len(lens)
        lens.append(int(rng.integers(512, 4096 + 1)))
        pars.append(-1)
        for _ in range(16):
            lens.append(int(rng.integers(128, 2048 + 1)))
            pars.append(root)
    tree = tree_from_preorder(lens, pars)
    return Workload("forest_small", "GRPO forest, 2 stars: prompts U[512,4096], 16 completions U[128,2048]; "
                    "32q/8kv, D=128", tree, 32, 8, 128, 0.5, 2, None, None)


def agent_tree_small() -> Workload:
    """The agent-tree recipe capped at 16,384 tokens."""
    rng = np.random.default_rng(3)
    tree = _random_tree(rng, lambda: _log_uniform(rng, 16, 4096), lambda: _log_uniform(rng, 16, 4096),
                        1, 4, 8, 16384)
    edge = np.nonzero(rng.random(tree.total_tokens) < 0.05)[0].astype(np.int32)
    return Workload("agent_small", "agent-call tree: 16384 tokens, depth<=8, branching U{1..4}, segments "
                    "logU[16,4096]; 32q/8kv, D=128", tree, 32, 8, 128, 0.5, 3, 4096, edge)


def long_fragment_small() -> Workload:
    """The long-fragment recipe scaled by 1/4 in its lengths (2K trunk, segments log-uniform in
    [64, 2048]), capped at 16,384 tokens, so that the tree still branches."""
    rng = np.random.default_rng(4)
    tree = _random_tree(rng, lambda: 2048, lambda: _log_uniform(rng, 64, 2048), 1, 3, 12, 16384)
    return Workload("long_small", "long bounded fragment: 16384 tokens, 2K trunk, depth<=12, branching U{1..3}, "
                    "segments logU[64,2048]; 64q/8kv, D=128", tree, 64, 8, 128, 0.5, 4, None, None)


CONFIGS: dict[str, Callable[[], Workload]] = {
    "tiny": tiny,
    "star": grpo_star,
    "forest": grpo_forest,
    "agent": agent_tree,
    "long": long_fragment,
    "forest_small": grpo_forest_small,
    "agent_small": agent_tree_small,
    "long_small": long_fragment_small,
}


def get(name: str) -> Workload:
    return CONFIGS[name]()


def _randn_chunked(gen, T: int, inner: tuple[int, ...]):
    import torch
    parts = []
    for t0 in range(0, T, CHUNK_TOKENS):
        n = min(CHUNK_TOKENS, T - t0)
        parts.append(torch.randn((n,) + inner, generator=gen, dtype=torch.float32))
    if not parts:
        return torch.empty((0,) + inner, dtype=torch.float32)
    return torch.cat(parts, 0)


def draw_tensors(w: Workload, dtype: str = "bf16", with_hidden: bool = False) -> dict:
    """Q, K, V, dO (and optionally the hidden tensor) as CPU torch tensors.

    ``dtype='bf16'`` rounds the scaled fp32 draws to bf16; ``'f32'`` keeps
    them in fp32.  Layouts: Q, dO ``[T, Hq, D]``; K, V ``[T, Hkv, D]``;
    hidden ``[T, hidden_dim]``.
    """
    import torch
    gen = torch.Generator("cpu")
    gen.manual_seed(w.seed)
    T, D = w.T, w.head_dim
    out = {}
    for name, heads in (("q", w.hq), ("k", w.hkv), ("v", w.hkv), ("do", w.hq)):
        x = _randn_chunked(gen, T, (heads, D))
        if name != "do":
            x.mul_(w.tensor_scale)
        out[name] = x.to(torch.bfloat16) if dtype == "bf16" else x
    if with_hidden and w.hidden_dim:
        h = _randn_chunked(gen, T, (w.hidden_dim,))
        out["hidden"] = h.to(torch.bfloat16) if dtype == "bf16" else h
    return out


# Vocabulary size for the sampled-edge vocabulary head.  The pages give none;
# 131,072 entries is a common size for large-vocabulary language models.
LM_HEAD_VOCAB = 131072


def draw_lm_head(num_actions: int, hidden_dim: int, vocab: int = LM_HEAD_VOCAB, seed: int = 0,
                 weight_scale: float = 2.0) -> dict:
    """Vocabulary-head weight, sampled labels and upstream gradients (CPU torch tensors).

    hidden_sel ``[num_actions, hidden_dim]`` bf16 ~ N(0, 1) (distributed like
    rows gathered from the workloads' hidden tensors); weight
    ``[vocab, hidden_dim]`` bf16 ~ N(0, 1) * weight_scale / sqrt(hidden_dim)
    (so logits have a standard deviation of about weight_scale); labels
    ``[num_actions]`` int32 uniform in [0, vocab); grad_logprob
    ``[num_actions]`` fp32 ~ N(0, 1).
    """
    import torch
    gen = torch.Generator("cpu")
    gen.manual_seed(seed)
    hidden_sel = _randn_chunked(gen, num_actions, (hidden_dim,))
    weight = _randn_chunked(gen, vocab, (hidden_dim,))
    weight.mul_(weight_scale / float(np.sqrt(hidden_dim)))
    labels = torch.randint(0, vocab, (num_actions,), generator=gen, dtype=torch.int64).to(torch.int32)
    grad = torch.randn(num_actions, generator=gen)
    return {"hidden_sel": hidden_sel.to(torch.bfloat16), "weight": weight.to(torch.bfloat16), "labels": labels,
            "grad_logprob": grad}


def random_small_tree(rng: np.random.Generator, max_segments: int = 8, max_len: int = 24,
                      forest: bool = True) -> Tree:
    """A small random preorder tree (or forest) for brute-force comparisons."""
    n = int(rng.integers(1, max_segments + 1))
    lens = [int(rng.integers(1, max_len + 1)) for _ in range(n)]
    parents = [-1]
    stack = [0]
    for s in range(1, n):
        # choose the parent among the current root path (or a new root)
        opts = list(stack) + ([-1] if forest else [])
        p = opts[int(rng.integers(0, len(opts)))]
        if p == -1:
            stack = []
        else:
            stack = stack[: stack.index(p) + 1]
        parents.append(p)
        stack.append(s)
    return tree_from_preorder(lens, parents)
