"""Seeded synthetic inputs for the MoE tree-verification layer.

This module is shared by the CUDA path (tests, bench) and by the oracle's tests.
It only draws random numbers and builds tree shapes; it holds none of the
method's arithmetic (no routing, no demand, no selection, no expert math).

Workload shapes follow the pages:
  * the draft tree is shaped like an EAGLE-3 tree with 5 draft steps, top-10
    expansion and 64 draft tokens ("AcceptMoE" article, section 03; "MoE and
    speculative decoding" blog, the chain-vs-tree section);
  * node hidden states are correlated along branches so that routing is
    correlated along a path (x_child = 0.8 x_parent + 0.6 N(0,1));
  * expert and router weights are i.i.d. N(0, std) rounded to the layer dtype.

Seeds: every generator takes an explicit integer seed. Trees use numpy's PCG64;
dense tensors use torch's generator on the requested device (Philox on CUDA,
mt19937 on the CPU), so the same seed on different devices gives different but
equally distributed values. Inputs a test compares across the two paths are
always generated once and handed to both.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

# ----------------------------------------------------------------------------
# Layer / workload configurations (sizes from the workloads the pages measure).
# ----------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class LayerShape:
    d: int          # hidden size
    E: int          # routed experts
    k: int          # experts per token (top-k)
    f: int          # SwiGLU intermediate size per expert
    dtype: str      # "fp32" or "bf16"

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "fp32" else 2

    @property
    def expert_bytes(self) -> int:
        """Bytes of one expert's W_gate + W_up + W_down."""
        return 3 * self.d * self.f * self.elem_bytes


TINY = LayerShape(d=256, E=16, k=2, f=128, dtype="fp32")
QWEN3_30B_A3B = LayerShape(d=2048, E=128, k=8, f=768, dtype="bf16")
GPT_OSS_120B = LayerShape(d=2880, E=128, k=4, f=2880, dtype="bf16")

# Commitment probability by draft depth (root = depth 0). The tiny case uses
# 0.7**depth; the Qwen/GPT-OSS workloads use the table below.
C_TINY = tuple(0.7 ** t for t in range(4))
C_EAGLE = (1.0, 0.8, 0.55, 0.35, 0.2, 0.1)

WEIGHT_STD = 0.02          # expert / router weights as the workloads state them
ROUTER_STD_PEAKED = 0.1    # labelled variant: a router whose demand is peaked


# ----------------------------------------------------------------------------
# Draft trees
# ----------------------------------------------------------------------------


@dataclasses.dataclass
class Tree:
    parent: np.ndarray   # int32 [N], parent[0] = -1, parent[n] < n
    depth: np.ndarray    # int32 [N], depth[0] = 0

    @property
    def N(self) -> int:
        return int(self.parent.shape[0])


def tiny_tree() -> Tree:
    """Root plus binary branching down to depth 3, 9 nodes in BFS order."""
    parent = np.array([-1, 0, 0, 1, 1, 2, 2, 3, 3], dtype=np.int32)
    return Tree(parent=parent, depth=_depths(parent))


def _depths(parent: np.ndarray) -> np.ndarray:
    depth = np.zeros(parent.shape[0], dtype=np.int32)
    for n in range(1, parent.shape[0]):
        depth[n] = depth[parent[n]] + 1
    return depth


@dataclasses.dataclass
class Candidates:
    parent: np.ndarray   # int32 [C], parent[0] = -1, parents before children
    depth: np.ndarray    # int32 [C]
    logp: np.ndarray     # float32 [C], cumulative draft log-probability (root 0)

    @property
    def C(self) -> int:
        return int(self.parent.shape[0])


def eagle_candidates(seed: int, steps: int = 5, topk: int = 10, vocab: int = 32,
                     alpha: float = 0.3) -> Candidates:
    """Every node an EAGLE-3-shaped expansion generates (the pool a drafter selects the
    verified tree from): `steps` steps, `topk` children per frontier node, the best
    `topk` new nodes form the next frontier. Same draws as eagle_tree for the same seed.
    Nodes in (depth, -logp) order, so parents come before children."""
    rng = np.random.Generator(np.random.PCG64(seed))
    par: List[int] = [-1]
    dep: List[int] = [0]
    lp: List[float] = [0.0]
    frontier = [0]
    for _ in range(steps):
        new: List[int] = []
        for p in frontier:
            probs = np.sort(rng.dirichlet(np.full(vocab, alpha)))[::-1][:topk]
            for q in probs:
                par.append(p)
                dep.append(dep[p] + 1)
                lp.append(lp[p] + math.log(max(float(q), 1e-300)))
                new.append(len(par) - 1)
        new.sort(key=lambda i: (-lp[i], i))
        frontier = new[:topk]
    order = [0] + sorted(range(1, len(par)), key=lambda i: (dep[i], -lp[i], i))
    remap = {old: new for new, old in enumerate(order)}
    parent = np.array([-1] + [remap[par[i]] for i in order[1:]], dtype=np.int32)
    return Candidates(parent=parent, depth=np.array([dep[i] for i in order], dtype=np.int32),
                      logp=np.array([lp[i] for i in order], dtype=np.float32))


def eagle_tree(seed: int, steps: int = 5, topk: int = 10, draft_tokens: int = 64,
               vocab: int = 32, alpha: float = 0.3) -> Tree:
    """An EAGLE-3-shaped draft tree: `steps` expansion steps, `topk` children per
    frontier node, the best `topk` new nodes form the next frontier, and the
    `draft_tokens` nodes with the highest cumulative draft log-probability are
    kept (plus the root). Draft probabilities of a node's children are the
    top-`topk` entries of a Dirichlet(alpha * 1_vocab) draw.

    Cumulative log-probability strictly decreases from parent to child, so the
    kept set is closed under ancestors. Nodes are returned in (depth, -logp)
    order, which puts every parent before its children.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    # node records: (parent_id, depth, cum_logp)
    par: List[int] = [-1]
    dep: List[int] = [0]
    lp: List[float] = [0.0]
    frontier = [0]
    for _ in range(steps):
        new: List[int] = []
        for p in frontier:
            probs = np.sort(rng.dirichlet(np.full(vocab, alpha)))[::-1][:topk]
            for q in probs:
                par.append(p)
                dep.append(dep[p] + 1)
                lp.append(lp[p] + math.log(max(float(q), 1e-300)))
                new.append(len(par) - 1)
        new.sort(key=lambda i: (-lp[i], i))
        frontier = new[:topk]
    cand = sorted(range(1, len(par)), key=lambda i: (-lp[i], i))[:draft_tokens]
    keep = [0] + sorted(cand, key=lambda i: (dep[i], -lp[i], i))
    remap = {old: new for new, old in enumerate(keep)}
    parent = np.array([-1] + [remap[par[i]] for i in keep[1:]], dtype=np.int32)
    depth = np.array([dep[i] for i in keep], dtype=np.int32)
    return Tree(parent=parent, depth=depth)


def tree_block(seed: int, B: int, kind: str = "eagle") -> Tuple[np.ndarray, np.ndarray]:
    """B independent trees stacked: parent/depth int32 [B, N] (tree-local parents)."""
    trees = [tiny_tree() if kind == "tiny" else eagle_tree(seed * 1009 + b) for b in range(B)]
    return (np.stack([t.parent for t in trees]).astype(np.int32),
            np.stack([t.depth for t in trees]).astype(np.int32))


# ----------------------------------------------------------------------------
# Dense tensors
# ----------------------------------------------------------------------------


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def hidden_states(seed: int, parent: np.ndarray, d: int, dtype: torch.dtype,
                  device="cpu", rho: float = 0.8) -> torch.Tensor:
    """Node hidden states [B*N, d]: root ~ N(0,1), child = rho*parent + sqrt(1-rho^2)*N(0,1).

    `parent` is [N] or [B, N] with tree-local parent indices."""
    par = np.atleast_2d(parent)
    B, N = par.shape
    g = _gen(seed, device)
    noise = torch.randn(B, N, d, generator=g, device=device, dtype=torch.float32)
    x = torch.empty_like(noise)
    s = math.sqrt(1.0 - rho * rho)
    for n in range(N):
        if n == 0:
            x[:, 0] = noise[:, 0]
        else:
            pidx = torch.as_tensor(par[:, n].astype(np.int64), device=device)
            x[:, n] = rho * x[torch.arange(B, device=device), pidx] + s * noise[:, n]
    return x.reshape(B * N, d).to(dtype).contiguous()


def router_weight(seed: int, shape: LayerShape, std: float = WEIGHT_STD, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    w = torch.randn(shape.E, shape.d, generator=g, device=device, dtype=torch.float32) * std
    return w.to(shape.torch_dtype).contiguous()


def expert_weights(seed: int, shape: LayerShape, std: float = WEIGHT_STD, device="cpu",
                   n_experts: Optional[int] = None):
    """(W_gate [E,f,d], W_up [E,f,d], W_down [E,d,f]) in the layer dtype, i.i.d. N(0,std).

    Generated one expert at a time in fp32 and rounded, so peak temporary memory
    is one expert."""
    E = shape.E if n_experts is None else n_experts
    dt = shape.torch_dtype
    g = _gen(seed, device)
    wg = torch.empty(E, shape.f, shape.d, device=device, dtype=dt)
    wu = torch.empty(E, shape.f, shape.d, device=device, dtype=dt)
    wd = torch.empty(E, shape.d, shape.f, device=device, dtype=dt)
    for e in range(E):
        for w in (wg, wu, wd):
            w[e].copy_(torch.randn(w.shape[1], w.shape[2], generator=g, device=device,
                                   dtype=torch.float32).mul_(std))
    return wg, wu, wd


def synthetic_logits(seed: int, parent: np.ndarray, E: int, scale: float = 1.0,
                     rho: float = 0.8) -> np.ndarray:
    """fp32 router-logit stand-ins [B*N, E] with the same branch correlation as
    the hidden states: root ~ N(0, scale^2), child = rho*parent + sqrt(1-rho^2)*noise."""
    par = np.atleast_2d(parent)
    B, N = par.shape
    rng = np.random.Generator(np.random.PCG64(seed))
    noise = rng.standard_normal((B, N, E)) * scale
    out = np.empty_like(noise)
    s = math.sqrt(1.0 - rho * rho)
    for n in range(N):
        out[:, n] = noise[:, n] if n == 0 else rho * out[np.arange(B), par[:, n]] + s * noise[:, n]
    return out.reshape(B * N, E).astype(np.float32)


def routing_from_sets(sets: Sequence[Sequence[int]], E: int) -> np.ndarray:
    """fp32 logits whose top-|set| per row is exactly the given expert set:
    chosen experts get 1.0, the rest 0.0, plus a small id-ordered offset so that
    no two logits in a row are equal."""
    L = np.zeros((len(sets), E), dtype=np.float64)
    for r, s in enumerate(sets):
        for e in s:
            L[r, e] = 1.0
    L -= 1e-3 * np.arange(E)[None, :]
    return L.astype(np.float32)


def random_assignments(seed: int, R: int, E: int, k: int, skew: float = 0.0) -> np.ndarray:
    """int32 [R, k] expert ids, distinct within a row. skew > 0 concentrates
    choices on low ids (a Zipf-like popularity), as a routing stress input."""
    rng = np.random.Generator(np.random.PCG64(seed))
    w = 1.0 / np.power(np.arange(1, E + 1), skew)
    w /= w.sum()
    out = np.empty((R, k), dtype=np.int32)
    for r in range(R):
        out[r] = rng.choice(E, size=k, replace=False, p=w)
    return out


def random_gates(seed: int, R: int, k: int) -> np.ndarray:
    """Positive fp32 weights [R, k] summing to 1 per row (a Dirichlet draw)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.dirichlet(np.ones(k), size=R).astype(np.float32)


def residency_mask(seed: int, E: int, resident: int) -> np.ndarray:
    """uint8 [E]: `resident` experts marked 1, chosen uniformly at random."""
    rng = np.random.Generator(np.random.PCG64(seed))
    m = np.zeros(E, dtype=np.uint8)
    m[rng.choice(E, size=resident, replace=False)] = 1
    return m
