"""ctypes wrapper around the plain-C oracle (moe_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package smoke check and
by the benchmark's CPU-baseline leg. The product path never imports it.

The wrapper only marshals numpy arrays into the C functions and composes them in
the layer's order (router -> top-k -> selection per tree -> permute -> experts ->
combine); all arithmetic is in moe_oracle.c.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import Dict, Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "libmoe_oracle.so")

NATURAL, ACCEPT, FIXED_B = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with plain gcc (no fast-math, no vectorisation flags, and no
    fused multiply-add contraction, so that fp32 steps round the same on x86 and Arm)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                        "-fvisibility=hidden", "-o", tmp, SRC, "-lm"], check=True)
        os.replace(tmp, LIB)
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        P = C.c_void_p
        i = C.c_int
        _lib.oracle_router.argtypes = [P, P, i, i, i, i, P]
        _lib.oracle_router.restype = None
        _lib.oracle_topk.argtypes = [P, i, i, i, P]
        _lib.oracle_topk.restype = C.c_double
        _lib.oracle_select_tree.argtypes = [P, P, i, i, i, P, i, i, i, i, i, P, i, i, i,
                                            P, P, P, P, P, P, P]
        _lib.oracle_select_tree.restype = i
        _lib.oracle_restricted_route.argtypes = [P, i, i, i, P, P, P]
        _lib.oracle_restricted_route.restype = None
        _lib.oracle_permute.argtypes = [P, i, i, i, P, P, P]
        _lib.oracle_permute.restype = None
        _lib.oracle_expert_ffn.argtypes = [P, i, P, P, P, i, i, i, P]
        _lib.oracle_expert_ffn.restype = None
        _lib.oracle_moe_combine.argtypes = [P, P, P, P, i, i, i, P, P, i, P, i, P]
        _lib.oracle_moe_combine.restype = None
        _lib.oracle_draft_select.argtypes = [i, i, i, P, P, P, C.c_float, i, P, P]
        _lib.oracle_draft_select.restype = i
        _lib.oracle_round_bf16.argtypes = [C.c_double]
        _lib.oracle_round_bf16.restype = C.c_uint16
        _lib.oracle_rmsnorm.argtypes = [P, i, i, i, C.c_double, P, P]
        _lib.oracle_rmsnorm.restype = None
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _raw(t):
    """A C-contiguous numpy view of a torch tensor or numpy array plus its dtype code
    (0 = fp32, 1 = bf16 as raw uint16 bits)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16), 1
            return t.to(torch.float32).numpy(), 0
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    if a.dtype == np.uint16:
        return a, 1
    return a.astype(np.float32, copy=False), 0


NORM_EPS = 1e-6


def round_bf16(v: float) -> int:
    """Raw bits of the bf16 nearest to v (ties to even)."""
    return int(lib().oracle_round_bf16(float(v)))


def rmsnorm(x, eps: float = NORM_EPS, unrounded: bool = False):
    """Pre-norm x / sqrt(mean(x^2) + eps) per row in fp64, rounded once to x's dtype:
    a uint16 array of bf16 bits for bf16 input (accepted by router / moe_combine as
    bf16), fp32 otherwise. With `unrounded`, also the fp64 values before rounding."""
    xa, dt = _raw(x)
    R, d = xa.shape
    out = np.empty((R, d), dtype=np.uint16 if dt == 1 else np.float32)
    x64 = np.empty((R, d), dtype=np.float64) if unrounded else None
    lib().oracle_rmsnorm(_p(xa), dt, R, d, eps, _p(x64), _p(out))
    return (out, x64) if unrounded else out


def router(x, Wr) -> np.ndarray:
    """fp64 router logits [R, E]."""
    xa, dt = _raw(x)
    wa, dt2 = _raw(Wr)
    assert dt == dt2
    R, d = xa.shape
    E = wa.shape[0]
    out = np.empty((R, E), dtype=np.float64)
    lib().oracle_router(_p(xa), _p(wa), dt, R, d, E, _p(out))
    return out


def topk(logits: np.ndarray, k: int):
    l = np.ascontiguousarray(logits, dtype=np.float32)
    R, E = l.shape
    idx = np.empty((R, k), dtype=np.int32)
    margin = lib().oracle_topk(_p(l), R, E, k, _p(idx))
    return idx, margin


def select_tree(logits: np.ndarray, depth: np.ndarray, k: int, c: Sequence[float],
                mode: int = ACCEPT, pool_all: bool = False, anchor: bool = True,
                prune: bool = False, resident: Optional[np.ndarray] = None,
                budget: int = 8, min_set: int = 16, fixed_B: int = 0) -> Dict:
    """Selection for one tree (demand, entropy and effective rank in fp64). Besides the
    choices it returns the demand D, the effective rank r (NaN outside ACCEPT) and the
    decision margins (see oracle_select_tree)."""
    l = np.ascontiguousarray(logits, dtype=np.float32)
    N, E = l.shape
    dep = np.ascontiguousarray(depth, dtype=np.int32)
    cc = np.ascontiguousarray(np.asarray(c, dtype=np.float64))
    res = None if resident is None else np.ascontiguousarray(resident, dtype=np.uint8)
    idx = np.empty((N, k), dtype=np.int32)
    gates = np.empty((N, k), dtype=np.float64)
    elig = np.empty(E, dtype=np.uint8)
    info = np.empty(4, dtype=np.int32)
    D = np.zeros(E, dtype=np.float64)
    margins = np.empty(5, dtype=np.float64)
    r = np.empty(1, dtype=np.float64)
    rc = lib().oracle_select_tree(_p(l), _p(dep), N, E, k, _p(cc), len(cc), mode,
                                  int(pool_all), int(anchor), int(prune), _p(res), budget,
                                  min_set, fixed_B, _p(idx), _p(gates), _p(elig), _p(info),
                                  _p(D), _p(margins), _p(r))
    if rc != 0:
        raise ValueError("oracle_select_tree: bad arguments")
    return dict(idx=idx, gates=gates, eligible=elig, union_nat=int(info[0]),
                union_sel=int(info[1]), m=int(info[2]), pruned=int(info[3]), D=D, r=float(r[0]),
                margin_topk=margins[0], margin_rank=margins[1], margin_fill=margins[2],
                margin_prune=margins[3], margin_restricted=margins[4])


def select_block(logits: np.ndarray, depth: np.ndarray, k: int, c: Sequence[float],
                 **kw) -> Dict:
    """Selection for B trees: logits [B*N, E], depth [B, N]. Per-tree results stacked."""
    dep = np.atleast_2d(depth)
    B, N = dep.shape
    outs = [select_tree(logits[b * N:(b + 1) * N], dep[b], k, c, **kw) for b in range(B)]
    res = dict(idx=np.concatenate([o["idx"] for o in outs]),
               gates=np.concatenate([o["gates"] for o in outs]),
               eligible=np.stack([o["eligible"] for o in outs]))
    for key in ("union_nat", "union_sel", "m", "pruned"):
        res[key] = np.array([o[key] for o in outs], dtype=np.int32)
    for key in ("margin_topk", "margin_rank", "margin_fill", "margin_prune", "margin_restricted"):
        res[key] = min(o[key] for o in outs)
    res["D"] = np.stack([o["D"] for o in outs])
    res["r"] = np.array([o["r"] for o in outs])
    res["trees"] = outs
    return res


def restricted_route(logits: np.ndarray, allowed: np.ndarray, k: int):
    """Each row's top-k among the experts with allowed[e] != 0 and its renormalised
    gates (the re-routing step on its own): (idx [R, k] int32, gates [R, k] fp64)."""
    l = np.ascontiguousarray(logits, dtype=np.float32)
    R, E = l.shape
    al = np.ascontiguousarray(np.asarray(allowed) != 0, dtype=np.uint8)
    if al.shape != (E,) or int(al.sum()) < k:
        raise ValueError("restricted_route: the mask needs E entries and at least k experts")
    idx = np.empty((R, k), dtype=np.int32)
    gates = np.empty((R, k), dtype=np.float64)
    lib().oracle_restricted_route(_p(l), R, E, k, _p(al), _p(idx), _p(gates))
    return idx, gates


def permute(idx: np.ndarray, E: int):
    a = np.ascontiguousarray(idx, dtype=np.int32)
    R, k = a.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(R * k, dtype=np.int32)
    lib().oracle_permute(_p(a), R, k, E, _p(counts), _p(offsets), _p(perm))
    return counts, offsets, perm


def expert_ffn(x_row: np.ndarray, e: int, Wg, Wu, Wd) -> np.ndarray:
    g, dt = _raw(Wg)
    u, _ = _raw(Wu)
    w, _ = _raw(Wd)
    E, f, d = g.shape
    xr = np.ascontiguousarray(x_row, dtype=np.float64)
    out = np.empty(d, dtype=np.float64)
    lib().oracle_expert_ffn(_p(xr), e, _p(g), _p(u), _p(w), dt, d, f, _p(out))
    return out


def moe_combine(x, Wg, Wu, Wd, idx: np.ndarray, gates: np.ndarray,
                rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """y [n_rows, d] (fp64) for the given routing."""
    xa, dt = _raw(x)
    g, dt2 = _raw(Wg)
    u, _ = _raw(Wu)
    w, _ = _raw(Wd)
    assert dt == dt2
    R, d = xa.shape
    f = g.shape[1]
    k = idx.shape[1]
    ia = np.ascontiguousarray(idx, dtype=np.int32)
    ga = np.ascontiguousarray(gates, dtype=np.float64)
    ra = None if rows is None else np.ascontiguousarray(np.asarray(rows), dtype=np.int32)
    n = R if rows is None else len(ra)
    y = np.empty((n, d), dtype=np.float64)
    lib().oracle_moe_combine(_p(xa), _p(g), _p(u), _p(w), dt, d, f, _p(ia), _p(ga), k, _p(ra),
                             n, _p(y))
    return y


def forward(x, Wr, Wg, Wu, Wd, depth: np.ndarray, k: int, c: Sequence[float],
            rows: Optional[Sequence[int]] = None, norm_input: bool = False,
            **select_kw) -> Dict:
    """The whole layer: (optionally the RMS pre-norm of x) -> router (fp64, rounded to
    fp32 for the decisions) -> per-tree selection -> permute -> gated expert outputs for
    `rows` (without the residual)."""
    if norm_input:
        x = rmsnorm(x)
    logits64 = router(x, Wr)
    l32 = logits64.astype(np.float32)
    E = l32.shape[1]
    sel = select_block(l32, depth, k, c, **select_kw)
    counts, offsets, perm = permute(sel["idx"], E)
    y = moe_combine(x, Wg, Wu, Wd, sel["idx"], sel["gates"], rows=rows)
    sel.update(logits=logits64, logits32=l32, counts=counts, offsets=offsets, perm=perm, y=y)
    return sel


def draft_select(parent: np.ndarray, logp: np.ndarray, footprint: np.ndarray, E: int,
                 lam: float, gamma: int):
    """Cost-aware draft selection: (selected node ids in selection order, |union|)."""
    par = np.ascontiguousarray(parent, dtype=np.int32)
    lp = np.ascontiguousarray(logp, dtype=np.float32)
    fp = np.ascontiguousarray(footprint, dtype=np.int32)
    n_cand, k = fp.shape
    sel = np.empty(max(gamma, 1), dtype=np.int32)
    nu = np.zeros(1, dtype=np.int32)
    n = lib().oracle_draft_select(n_cand, k, E, _p(par), _p(lp), _p(fp), float(lam), gamma,
                                  _p(sel), _p(nu))
    return sel[:n].copy(), int(nu[0])
