"""GPU parity: every step of the CUDA path, called through the C ABI, against the
CPU oracle on the same seeded inputs.

Bars: expert indices, eligible sets, set sizes, per-expert counts and the
permutation are bit-exact given the same fp32 router logits; router logits within
1e-4 of the row's largest |logit|; gates within 1e-6; bf16 layer outputs within
2e-2 * max|ref| (fp32 layers within 1e-4 * max|ref|).

Decisions are compared with the oracle's fp64 definition of demand, entropy and
effective rank. The device decides in fp32 when its rounding bound certifies the
result and recomputes the tree in fp64 otherwise, so every tree must match. Only a
tree whose fp64 decision margin is below TIE64 (1e-11, where CUDA's and the C
library's fp64 exp and the two summation orders may disagree) is excused from the
exact comparison; for such a tree the test checks that the device's answer is one
of the valid ones (a size the margins allow, a demand-ordered fill, and the
restricted top-k over the device's own eligible set).
"""
import math

import numpy as np
import pytest
import torch

from expert_select_gb300 import moetree as M
from expert_select_gb300 import workload as W
from oracle import oracle as O

pytestmark = pytest.mark.gpu

TIE64 = 1e-11
DEV = "cuda"
NF = M.MOE_INFO_FIELDS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from expert_select_gb300 import build
    build.build()
    M.lib()


def _sync():
    torch.cuda.synchronize()


def _desc(shape):
    return M.layer_desc(shape.d, shape.E, shape.k, shape.f, shape.dtype)


def _tol(shape):
    return 2e-2 if shape.dtype == "bf16" else 1e-4


def _assert_close_rows(got, ref, shape):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref).max()
    assert err <= _tol(shape) * np.abs(ref).max(), (err, np.abs(ref).max())


def _select_gpu(shape, P, logits, depth, B, N, resident=None):
    L = _desc(shape)
    R = B * N
    lg = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(DEV)
    dp = torch.from_numpy(np.ascontiguousarray(depth.reshape(-1).astype(np.int32))).to(DEV)
    idx = torch.empty(R, shape.k, dtype=torch.int32, device=DEV)
    gates = torch.empty(R, shape.k, dtype=torch.float32, device=DEV)
    elig = torch.empty(B, shape.E, dtype=torch.uint8, device=DEV)
    info = torch.empty(B, NF, dtype=torch.int32, device=DEV)
    res = None if resident is None else torch.from_numpy(resident).to(DEV)
    M.moe_tree_select(L, P, lg, dp, B, N, res, idx, gates, elig, info)
    _sync()
    return idx.cpu().numpy(), gates.cpu().numpy(), elig.cpu().numpy(), info.cpu().numpy()


def _fp64_tied(o):
    return min(o["margin_rank"], o["margin_fill"], o["margin_prune"]) < TIE64


def _check_valid(shape, kw, l, o, gidx, ggates, gelig_b, ginfo_b):
    """A valid selection for a tree whose fp64 margins tie: the size is one the rank
    margin allows, the anchor is in, the fill is demand-ordered up to the tie, pruned
    experts are non-resident non-anchor members, and the routing is the restricted
    top-k over the device's own eligible set."""
    k = shape.k
    S = set(np.flatnonzero(gelig_b).tolist())
    nat, _ = O.topk(l[:1], k)
    A = set(nat[0].tolist()) if kw.get("anchor", True) else set()
    assert A <= S
    m_ok = {o["m"]} if o["margin_rank"] >= TIE64 else {o["m"] - 1, o["m"], o["m"] + 1}
    assert ginfo_b[2] in m_ok and ginfo_b[2] >= k
    D = o["D"]
    pool = set(range(shape.E)) if kw.get("pool_all") else set(O.topk(l, k)[0].ravel().tolist())
    if not kw.get("prune"):
        assert len(S) == ginfo_b[2]
        inside, outside = S - A, (pool - A) - S
        if inside and outside:
            assert min(D[e] for e in inside) >= max(D[e] for e in outside) * (1 - 1e-9)
    else:
        assert ginfo_b[3] <= kw.get("budget", 8)
        assert len(S) == ginfo_b[2] - ginfo_b[3]
    ridx, rg = O.restricted_route(l, gelig_b, k)
    np.testing.assert_array_equal(gidx, ridx)
    np.testing.assert_allclose(ggates, rg, atol=1e-6)


def _check_selection(shape, kw, logits, depth, gidx, ggates, gelig, ginfo, N, B):
    """Compares one block's selection tree by tree with the fp64 oracle; returns the
    number of trees excused as fp64 ties (validity-checked instead)."""
    tied = 0
    okw = {k: v for k, v in kw.items() if k != "c"}
    for b in range(B):
        sl = slice(b * N, (b + 1) * N)
        o = O.select_tree(logits[sl], depth[b], shape.k, kw["c"], **okw)
        if _fp64_tied(o):
            tied += 1
            _check_valid(shape, kw, logits[sl], o, gidx[sl], ggates[sl], gelig[b], ginfo[b])
            continue
        np.testing.assert_array_equal(gelig[b], o["eligible"])
        np.testing.assert_array_equal(gidx[sl], o["idx"])
        np.testing.assert_allclose(ggates[sl], o["gates"], atol=1e-6)
        assert ginfo[b, :4].tolist() == [o["union_nat"], o["union_sel"], o["m"], o["pruned"]]
        if kw["mode"] == O.NATURAL:
            assert ginfo[b, 4] == 0
    return tied


# ------------------------------------------------------------------- router

ROUTER_E256 = W.LayerShape(d=512, E=256, k=8, f=128, dtype="bf16")
ROUTER_E64 = W.LayerShape(d=320, E=64, k=4, f=128, dtype="bf16")


# R >= 192 (bf16) runs on the tensor cores: 32-row tiles, 64-row tiles past 152 x 32
# rows, two 128-expert tiles for E = 256, zero-filled router rows for E = 64.
@pytest.mark.parametrize("shape,R", [(W.TINY, 9), (W.TINY, 1), (W.QWEN3_30B_A3B, 65),
                                     (W.QWEN3_30B_A3B, 37), (W.QWEN3_30B_A3B, 191),
                                     (W.QWEN3_30B_A3B, 192), (W.QWEN3_30B_A3B, 411),
                                     (W.QWEN3_30B_A3B, 4160), (W.QWEN3_30B_A3B, 9797),
                                     (W.GPT_OSS_120B, 65), (W.GPT_OSS_120B, 333),
                                     (ROUTER_E256, 500), (ROUTER_E64, 200)])
def test_router_logits(shape, R):
    chain = np.arange(-1, R - 1, dtype=np.int32)
    x = W.hidden_states(11 + R, chain, shape.d, shape.torch_dtype)
    wr = W.router_weight(12, shape, std=0.1)
    logits = torch.empty(R, shape.E, dtype=torch.float32, device=DEV)
    M.moe_router_logits(_desc(shape), x.to(DEV), wr.to(DEV), logits)
    _sync()
    rows = np.arange(R) if R <= 130 else np.random.default_rng(0).choice(R, 130, replace=False)
    ref = O.router(x[rows], wr)
    got = logits.cpu().numpy()[rows]
    scale = np.abs(ref).max(axis=1, keepdims=True)
    assert (np.abs(got - ref) <= 1e-4 * scale).all()


# ---------------------------------------------------------------- selection

SELECT_CASES = [
    # (id, shape, B, tree kind, logit scale, select kwargs)
    ("tiny-nat", W.TINY, 1, "tiny", 1.0, dict(mode=O.NATURAL)),
    ("tiny-acc", W.TINY, 3, "tiny", 3.0, dict(mode=O.ACCEPT)),
    ("tiny-fixB", W.TINY, 2, "tiny", 3.0, dict(mode=O.FIXED_B, fixed_B=5)),
    ("qwen-acc-flat", W.QWEN3_30B_A3B, 1, "eagle", 1.0, dict(mode=O.ACCEPT)),
    ("qwen-acc-peaked", W.QWEN3_30B_A3B, 4, "eagle", 4.5, dict(mode=O.ACCEPT)),
    ("qwen-nat", W.QWEN3_30B_A3B, 2, "eagle", 4.5, dict(mode=O.NATURAL)),
    ("qwen-pool-all", W.QWEN3_30B_A3B, 2, "eagle", 4.5, dict(mode=O.ACCEPT, pool_all=True)),
    ("qwen-no-anchor", W.QWEN3_30B_A3B, 2, "eagle", 4.5, dict(mode=O.FIXED_B, fixed_B=20,
                                                             anchor=False)),
    ("gptoss-prune", W.GPT_OSS_120B, 4, "eagle", 4.5, dict(mode=O.ACCEPT, prune=True,
                                                           budget=8, min_set=16)),
    ("gptoss-prune-tight", W.GPT_OSS_120B, 2, "eagle", 4.5, dict(mode=O.ACCEPT, prune=True,
                                                                 budget=30, min_set=4)),
    ("e256-k16", W.LayerShape(d=64, E=256, k=16, f=64, dtype="fp32"), 2, "eagle", 3.0,
     dict(mode=O.ACCEPT)),
]


@pytest.mark.parametrize("case", SELECT_CASES, ids=[c[0] for c in SELECT_CASES])
def test_selection_bit_exact(case):
    _, shape, B, kind, scale, kw = case
    kw = dict(kw)
    c = W.C_TINY if kind == "tiny" else W.C_EAGLE
    parent, depth = W.tree_block(101 + B, B, kind)
    N = parent.shape[1]
    logits = W.synthetic_logits(202 + B, parent, shape.E, scale)
    resident = W.residency_mask(7, shape.E, 48) if kw.get("prune") else None
    mode = {O.NATURAL: M.MOE_ROUTE_NATURAL, O.ACCEPT: M.MOE_ROUTE_ACCEPT,
            O.FIXED_B: M.MOE_ROUTE_FIXED_B}[kw["mode"]]
    P = M.select_params(mode, c, pool_all=kw.get("pool_all", False),
                        anchor=kw.get("anchor", True), prune=kw.get("prune", False),
                        reroute_budget=kw.get("budget", 8), min_set=kw.get("min_set", 16),
                        fixed_B=kw.get("fixed_B", 0))
    gidx, gg, ge, gi = _select_gpu(shape, P, logits, depth, B, N, resident)
    okw = dict(kw, c=c)
    if resident is not None:
        okw["resident"] = resident
    tied = _check_selection(shape, okw, logits, depth, gidx, gg, ge, gi, N, B)
    assert tied == 0  # no fp64 ties on these seeded trees: every tree compared exactly


# ------------------------------------------- near ties: the fp64 pass of the selector

def _tree_of(N, seed):
    """An EAGLE-3-shaped 65-node tree, or a random tree of N nodes (N > 256 takes the
    one-CTA selector)."""
    if N == 65:
        t = W.eagle_tree(seed)
        return t.parent, t.depth
    rng = np.random.default_rng(seed)
    parent = np.array([-1] + [int(rng.integers(0, n)) for n in range(1, N)], np.int32)
    depth = np.zeros(N, np.int32)
    for n in range(1, N):
        depth[n] = depth[parent[n]] + 1
    return parent, depth


def _tie_columns(l, D, keep, copy, up):
    """Expert `copy` gets expert `keep`'s logits at every node, then one fp32 ulp up (or
    down) at the node where `keep` weighs most: the two demands then differ by ~1e-8
    relative, below what fp32 resolves and far above fp64's rounding."""
    l2 = l.copy()
    l2[:, copy] = l2[:, keep]
    n0 = int(np.argmax(l[:, keep] - l.max(axis=1)))
    l2[n0, copy] = np.nextafter(l2[n0, keep], np.float32(np.inf if up else -np.inf))
    return l2


def _near_tie_fill(l, depth, k, c, kw):
    """Moves the fill cut onto a near-tie (pool = all experts, so the natural union does
    not move with the edit); returns logits whose fp64 fill margin is below 1e-6."""
    for _ in range(8):
        o = O.select_tree(l, depth, k, c, **kw)
        if 1e-11 < o["margin_fill"] < 1e-6:
            return l, o
        A = set(O.topk(l[:1], k)[0][0].tolist())
        cand = sorted(set(range(l.shape[1])) - A, key=lambda e: (-o["D"][e], e))
        F = o["m"] - k
        l = _tie_columns(l, o["D"], cand[F - 1], cand[F], up=False)
    pytest.fail("could not build a fill near-tie")


@pytest.mark.parametrize("E,N,mode", [(32, 65, O.FIXED_B), (128, 65, O.ACCEPT),
                                      (256, 65, O.FIXED_B), (64, 300, O.ACCEPT)])
def test_fp64_pass_decides_a_fill_near_tie(E, N, mode):
    """Two experts whose demands differ by ~1e-8 sit on either side of the fill cut: the
    fp32 pass cannot order them, takes the fp64 pass (info[4] = 1), and the eligible set
    equals the fp64 oracle's."""
    shape = W.LayerShape(d=64, E=E, k=4, f=64, dtype="fp32")
    parent, depth = _tree_of(N, 7 + E)
    l = W.synthetic_logits(8 + E, parent[None], E, 3.0)
    kw = dict(mode=mode, pool_all=True, fixed_B=14)
    l, o = _near_tie_fill(l, depth, shape.k, W.C_EAGLE, kw)
    omode = {O.ACCEPT: M.MOE_ROUTE_ACCEPT, O.FIXED_B: M.MOE_ROUTE_FIXED_B}[mode]
    P = M.select_params(omode, W.C_EAGLE, pool_all=True, fixed_B=14)
    gidx, gg, ge, gi = _select_gpu(shape, P, l, depth[None], 1, N)
    assert gi[0, 4] == 1
    assert _check_selection(shape, dict(kw, c=W.C_EAGLE), l, depth[None], gidx, gg, ge, gi,
                            N, 1) == 0


@pytest.mark.parametrize("E,N", [(64, 65), (64, 300)])
def test_fp64_pass_decides_a_prune_near_tie(E, N):
    """The last expert pruning removes and the next one differ by ~1e-8 in demand."""
    shape = W.LayerShape(d=64, E=E, k=4, f=64, dtype="fp32")
    parent, depth = _tree_of(N, 30 + N)
    l = W.synthetic_logits(31 + N, parent[None], E, 3.0)
    res = W.residency_mask(5, E, E // 2)
    kw = dict(mode=O.FIXED_B, pool_all=True, fixed_B=24, prune=True, resident=res, budget=3,
              min_set=4)
    for _ in range(8):
        o = O.select_tree(l, depth, shape.k, W.C_EAGLE, **kw)
        if 1e-11 < o["margin_prune"] < 1e-6:
            break
        base = O.select_tree(l, depth, shape.k, W.C_EAGLE, **dict(kw, prune=False))
        A = set(O.topk(l[:1], shape.k)[0][0].tolist())
        S = set(np.flatnonzero(base["eligible"]).tolist())
        rem = sorted([e for e in S - A if not res[e]], key=lambda e: (base["D"][e], e))
        r = o["pruned"]
        assert 0 < r < len(rem)
        l = _tie_columns(l, base["D"], rem[r - 1], rem[r], up=True)
    else:
        pytest.fail("could not build a prune near-tie")
    P = M.select_params(M.MOE_ROUTE_FIXED_B, W.C_EAGLE, pool_all=True, fixed_B=24, prune=True,
                        reroute_budget=3, min_set=4)
    gidx, gg, ge, gi = _select_gpu(shape, P, l, depth[None], 1, N, res)
    assert gi[0, 4] == 1
    assert _check_selection(shape, dict(kw, c=W.C_EAGLE), l, depth[None], gidx, gg, ge, gi,
                            N, 1) == 0


@pytest.mark.parametrize("E,N,side", [(128, 65, 1.0), (128, 65, -1.0), (64, 300, 1.0)])
def test_fp64_pass_decides_a_size_near_integer(E, N, side):
    """Logits scaled so that exp(H) lies 4e-8 (relative) above an integer n (set size
    n + 1: beyond the 1e-9 snap) or below it (size n): fp32 cannot tell, fp64 can."""
    shape = W.LayerShape(d=64, E=E, k=4, f=64, dtype="fp32")
    parent, depth = _tree_of(N, 50 + N)
    base = W.synthetic_logits(51 + N, parent[None], E, 3.0).astype(np.float64)
    kw = dict(mode=O.ACCEPT, pool_all=True)
    r_of = lambda a: O.select_tree((base * a).astype(np.float32), depth, shape.k,  # noqa: E731
                                   W.C_EAGLE, **kw)["r"]
    n = round(r_of(1.0))
    target = n * (1.0 + side * 4e-8)
    lo, hi = 0.7, 1.4  # exp(H) falls as the logits sharpen
    assert r_of(lo) > target > r_of(hi)
    for _ in range(80):
        mid = 0.5 * (lo + hi)
        if r_of(mid) > target:
            lo = mid
        else:
            hi = mid
    l = (base * lo).astype(np.float32)
    o = O.select_tree(l, depth, shape.k, W.C_EAGLE, **kw)
    assert 1e-11 < o["margin_rank"] < 1e-6 and abs(o["r"] / n - 1) < 1e-6
    assert o["m"] == (n + 1 if side > 0 else n)
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE, pool_all=True)
    gidx, gg, ge, gi = _select_gpu(shape, P, l, depth[None], 1, N)
    assert gi[0, 4] == 1
    assert _check_selection(shape, dict(kw, c=W.C_EAGLE), l, depth[None], gidx, gg, ge, gi,
                            N, 1) == 0


@pytest.mark.parametrize("scale", [20.0, 40.0])
def test_wide_logit_ranges(scale):
    """Logit ranges of 150-300 within a node (as deep in a residual stack of layers): the
    far tails of each softmax underflow in fp32, which the certificate bounds in absolute
    terms. Every tree matches the fp64 oracle, and the fp32 pass still decides most."""
    shape = W.QWEN3_30B_A3B
    B = 16
    parent, depth = W.tree_block(616, B, "eagle")
    N = parent.shape[1]
    logits = W.synthetic_logits(617, parent, shape.E, scale)
    assert float((logits.max(1) - logits.min(1)).max()) > 150
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    gidx, gg, ge, gi = _select_gpu(shape, P, logits, depth, B, N)
    assert _check_selection(shape, dict(mode=O.ACCEPT, c=W.C_EAGLE), logits, depth, gidx, gg,
                            ge, gi, N, B) == 0
    assert gi[:, 4].sum() <= B // 2, gi[:, 4]


def test_fp32_certificate_decides_ordinary_trees():
    """64 peaked EAGLE-3-shaped trees (set sizes in the pages' 23-34 range): all match the
    fp64 oracle and the fp32 pass decides nearly all of them on its own."""
    shape = W.QWEN3_30B_A3B
    parent, depth = W.tree_block(606, 64, "eagle")
    N = parent.shape[1]
    logits = W.synthetic_logits(607, parent, shape.E, 4.5)
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    gidx, gg, ge, gi = _select_gpu(shape, P, logits, depth, 64, N)
    assert _check_selection(shape, dict(mode=O.ACCEPT, c=W.C_EAGLE), logits, depth, gidx, gg,
                            ge, gi, N, 64) == 0
    assert gi[:, 4].sum() <= 3, gi[:, 4].sum()


def test_selection_large_tree_single_cta_path():
    """Trees of more than 256 nodes take the one-CTA selector; 300- and 1000-node random
    trees, AcceptMoE and pruning, against the oracle."""
    shape = W.LayerShape(d=64, E=64, k=4, f=64, dtype="fp32")
    for N, seed in ((300, 1), (1000, 2)):
        rng = np.random.default_rng(seed)
        parent = np.array([-1] + [int(rng.integers(0, n)) for n in range(1, N)], np.int32)
        depth = np.zeros(N, np.int32)
        for n in range(1, N):
            depth[n] = depth[parent[n]] + 1
        logits = W.synthetic_logits(seed, parent, shape.E, 3.0)
        res = W.residency_mask(seed, shape.E, 20)
        P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE, prune=True, reroute_budget=8,
                            min_set=6)
        gidx, gg, ge, gi = _select_gpu(shape, P, logits, depth[None], 1, N, res)
        tied = _check_selection(shape, dict(mode=O.ACCEPT, prune=True, budget=8, min_set=6,
                                            resident=res, c=W.C_EAGLE),
                                logits, depth[None], gidx, gg, ge, gi, N, 1)
        assert tied == 0


@pytest.mark.parametrize("B,N,E,k", [(1, 411, 128, 8), (3, 1000, 64, 4), (2, 3000, 256, 16),
                                     (64, 65, 128, 8), (1, 1, 40, 3), (5, 129, 40, 1)])
def test_selection_natural_any_tree_size(B, N, E, k):
    """Natural routing runs one cluster per tree with a warp per node, for any N."""
    shape = W.LayerShape(d=64, E=E, k=k, f=64, dtype="fp32")
    rng = np.random.default_rng(N + B)
    parent = np.full((B, N), -1, np.int32)
    for b in range(B):
        parent[b, 1:] = [int(rng.integers(0, n)) for n in range(1, N)]
    depth = np.zeros((B, N), np.int32)
    for b in range(B):
        for n in range(1, N):
            depth[b, n] = depth[b, parent[b, n]] + 1
    logits = W.synthetic_logits(N + 7 * B, parent, E, 3.0)
    P = M.select_params(M.MOE_ROUTE_NATURAL, [1.0])
    gidx, gg, ge, gi = _select_gpu(shape, P, logits, depth, B, N)
    tied = _check_selection(shape, dict(mode=O.NATURAL, c=[1.0]), logits, depth, gidx, gg, ge,
                            gi, N, B)
    assert tied == 0


def test_selection_root_only_and_all_experts():
    # N = 1: the root alone; E = k: every expert is chosen by every node
    for shape, N in ((W.LayerShape(d=64, E=16, k=2, f=64, dtype="fp32"), 1),
                     (W.LayerShape(d=64, E=4, k=4, f=64, dtype="fp32"), 9)):
        depth = np.zeros((1, N), dtype=np.int32) if N == 1 else W.tiny_tree().depth[None]
        parent = np.full((1, N), -1, np.int32) if N == 1 else W.tiny_tree().parent[None]
        logits = W.synthetic_logits(5, parent, shape.E, 2.0)
        P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_TINY)
        gidx, gg, ge, gi = _select_gpu(shape, P, logits, depth, 1, N)
        o = O.select_tree(logits, depth[0], shape.k, W.C_TINY)
        np.testing.assert_array_equal(gidx, o["idx"])
        np.testing.assert_array_equal(ge[0], o["eligible"])
        assert gi[0, :4].tolist() == [o["union_nat"], o["union_sel"], o["m"], o["pruned"]]


def test_worked_examples_through_device():
    """The blog's two routing examples, routed and grouped by the device kernels."""
    shape = W.LayerShape(d=64, E=16, k=2, f=64, dtype="fp32")
    L = _desc(shape)
    for sets, union, counts in (([[2, 7], [2, 7], [2, 9], [4, 11]], 5,
                                 {2: 3, 7: 2, 9: 1, 4: 1, 11: 1}),
                                ([[1, 3], [6, 7], [1, 8], [4, 9], [2, 10]], 9, {1: 2, 3: 1})):
        logits = W.routing_from_sets(sets, 16)
        N = len(sets)
        P = M.select_params(M.MOE_ROUTE_NATURAL, [1.0])
        gidx, _, _, gi = _select_gpu(shape, P, logits, np.zeros((1, N), np.int32), 1, N)
        assert gi[0, 0] == union
        idx = torch.from_numpy(gidx).to(DEV)
        cnt = torch.empty(16, dtype=torch.int32, device=DEV)
        off = torch.empty(17, dtype=torch.int32, device=DEV)
        perm = torch.empty(N * 2, dtype=torch.int32, device=DEV)
        ws = M.workspace(L, 1, N)
        M.moe_expert_permute(L, idx, cnt, off, perm, ws)
        _sync()
        c = cnt.cpu().numpy()
        assert int((c > 0).sum()) == union
        for e, v in counts.items():
            assert c[e] == v
        # the block counters: union, assignments and reuse = 1 - union / assignments
        st = M.moe_tree_block_stats(L, 1, N, torch.from_numpy(gi).to(DEV), cnt)
        assert (st.union_experts, st.assignments, st.trees) == (union, 2 * N, 1)
        assert st.reuse == pytest.approx(1 - union / (2 * N))
        assert st.max_per_expert == max(counts.values())
        assert st.union_nat_mean == st.union_sel_mean == union and st.exact_trees == 0


def test_tree_route_equals_router_then_select():
    """moe_tree_route (hidden states in) gives bit for bit what moe_router_logits followed
    by moe_tree_select give, and the selection equals the fp64 oracle's on those logits;
    the block counters read from the workspace match the forward call's outputs."""
    shape = W.QWEN3_30B_A3B
    B = 4
    parent, depth = W.tree_block(515, B, "eagle")
    N = parent.shape[1]
    R = B * N
    x = W.hidden_states(516, parent, shape.d, torch.bfloat16).to(DEV)
    wr = W.router_weight(517, shape, std=0.1, device=DEV)
    L = _desc(shape)
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    dp = torch.from_numpy(depth.reshape(-1).copy()).to(DEV)
    outs = []
    for fused in (True, False):
        lg = torch.empty(R, shape.E, device=DEV)
        idx = torch.empty(R, shape.k, dtype=torch.int32, device=DEV)
        g = torch.empty(R, shape.k, device=DEV)
        el = torch.empty(B, shape.E, dtype=torch.uint8, device=DEV)
        inf = torch.empty(B, NF, dtype=torch.int32, device=DEV)
        if fused:
            M.moe_tree_route(L, P, x, wr, dp, B, N, None, lg, idx, g, el, inf)
        else:
            M.moe_router_logits(L, x, wr, lg)
            M.moe_tree_select(L, P, lg, dp, B, N, None, idx, g, el, inf)
        _sync()
        outs.append([t.cpu().numpy() for t in (lg, idx, g, el, inf)])
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)
    lg, idx, g, el, inf = outs[0]
    assert _check_selection(shape, dict(mode=O.ACCEPT, c=W.C_EAGLE), lg, depth, idx, g, el, inf,
                            N, B) == 0
    # the same block through the whole layer, counters read back from the workspace
    wg, wu, wd = _weights(shape, 518)
    ws = M.workspace(L, B, N)
    y = torch.empty(R, shape.d, dtype=torch.bfloat16, device=DEV)
    M.moe_tree_forward(L, P, x, wr, wg, wu, wd, None, dp, B, N, None, y, ws)
    st = M.moe_tree_block_stats(L, B, N, ws=ws)
    cnt = np.bincount(idx.ravel(), minlength=shape.E)
    assert st.assignments == R * shape.k and st.union_experts == int((cnt > 0).sum())
    assert st.max_per_expert == int(cnt.max())
    assert st.union_sel_mean == pytest.approx(inf[:, 1].mean())
    assert st.m_mean == pytest.approx(inf[:, 2].mean())
    assert st.reuse == pytest.approx(1 - st.union_experts / st.assignments)


# ------------------------------------------------------------------ permute

# The last four: row-block masks and prefixes that would not fit in one CTA's shared memory
# (E = 256 past ~3570 rows), built by the many-CTA mask kernel and scanned in place, both
# below and above 8192 assignments, and a block that still fits beside them.
@pytest.mark.parametrize("R,E,k,skew", [(1, 16, 2, 0.0), (9, 16, 2, 0.0), (65, 128, 8, 0.0),
                                        (65, 128, 8, 1.5), (520, 128, 4, 1.0),
                                        (4160, 128, 8, 0.8), (33, 256, 16, 0.5),
                                        (200, 256, 16, 0.7), (7000, 128, 8, 0.3),
                                        (2100, 256, 2, 0.0), (5000, 256, 1, 0.0),
                                        (3600, 256, 5, 0.4), (20000, 256, 2, 0.2)])
def test_permute_bit_exact(R, E, k, skew):
    shape = W.LayerShape(d=64, E=E, k=k, f=64, dtype="fp32")
    L = _desc(shape)
    idx = W.random_assignments(31 + R, R, E, k, skew)
    cnt = torch.empty(E, dtype=torch.int32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(R * k, dtype=torch.int32, device=DEV)
    ws = M.workspace(L, 1, R)
    M.moe_expert_permute(L, torch.from_numpy(idx).to(DEV), cnt, off, perm, ws)
    _sync()
    rc, ro, rp = O.permute(idx, E)
    np.testing.assert_array_equal(cnt.cpu().numpy(), rc)
    np.testing.assert_array_equal(off.cpu().numpy(), ro)
    np.testing.assert_array_equal(perm.cpu().numpy(), rp)
    assert M.moe_workspace_check(ws) == 0


def test_permute_flags_bad_and_duplicate_ids():
    shape = W.LayerShape(d=64, E=16, k=2, f=64, dtype="fp32")
    L = _desc(shape)
    idx = np.array([[1, 2], [3, 99], [4, 4], [5, -1]], dtype=np.int32)
    cnt = torch.empty(16, dtype=torch.int32, device=DEV)
    off = torch.empty(17, dtype=torch.int32, device=DEV)
    perm = torch.empty(8, dtype=torch.int32, device=DEV)
    ws = M.workspace(L, 1, 4)
    M.moe_expert_permute(L, torch.from_numpy(idx).to(DEV), cnt, off, perm, ws)
    _sync()
    c = cnt.cpu().numpy()
    assert c.sum() == 5 and c[4] == 1
    assert perm.cpu().numpy()[:5].tolist() == [0, 1, 2, 4, 6]
    assert M.moe_workspace_check(ws) & 1
    assert M.moe_workspace_check(ws) == 0  # cleared by the read


@pytest.mark.parametrize("R,k", [(1000, 4), (4160, 8), (700, 3)])
def test_permute_large_blocks_with_bad_and_repeated_ids(R, k):
    """Blocks past 2048 assignments place a row's choices from one thread; a repeated
    expert keeps its first slot and ids outside [0, E) are dropped, as in small blocks.
    Expected: the valid first-occurrence assignments sorted by (expert, row, slot)."""
    E = 64
    shape = W.LayerShape(d=64, E=E, k=k, f=64, dtype="fp32")
    L = _desc(shape)
    idx = W.random_assignments(900 + R, R, E, k, 0.5)
    rng = np.random.default_rng(R)
    for r in rng.choice(R, 40, replace=False):
        idx[r, k - 1] = idx[r, 0]            # a repeated expert
    for r in rng.choice(R, 40, replace=False):
        idx[r, int(rng.integers(0, k))] = int(rng.choice([-3, E, E + 7]))
    keep = []
    for r in range(R):
        seen = set()
        for j in range(k):
            e = int(idx[r, j])
            if 0 <= e < E and e not in seen:
                keep.append((e, r, j))
            seen.add(e)
    keep.sort()
    cnt = torch.empty(E, dtype=torch.int32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(R * k, dtype=torch.int32, device=DEV)
    ws = M.workspace(L, 1, R)
    M.moe_expert_permute(L, torch.from_numpy(idx).to(DEV), cnt, off, perm, ws)
    _sync()
    ref_perm = [r * k + j for _, r, j in keep]
    got = perm.cpu().numpy()
    assert got[:len(ref_perm)].tolist() == ref_perm
    assert (got[len(ref_perm):] == -1).all()
    ref_cnt = np.bincount([e for e, _, _ in keep], minlength=E)
    np.testing.assert_array_equal(cnt.cpu().numpy(), ref_cnt)
    np.testing.assert_array_equal(off.cpu().numpy(), np.concatenate([[0], np.cumsum(ref_cnt)]))
    assert M.moe_workspace_check(ws) & 1


# ------------------------------------------------------------- expert math

def _weights(shape, seed, device=DEV, E=None):
    return W.expert_weights(seed, shape, device=device, n_experts=E)


GPTOSS32 = W.LayerShape(d=2880, E=32, k=4, f=2880, dtype="bf16")
SMALL_BF16 = W.LayerShape(d=256, E=16, k=2, f=128, dtype="bf16")

EXPERT_CASES = [
    ("tiny-simt", W.TINY, 9, 0.0, M.MOE_FFN_SIMT, None),
    ("tiny-ragged", W.TINY, 23, 1.2, M.MOE_FFN_SIMT, None),
    ("qwen-simt", W.QWEN3_30B_A3B, 65, 1.0, M.MOE_FFN_SIMT, 24),
    ("gptoss-simt", GPTOSS32, 65, 0.7, M.MOE_FFN_SIMT, 24),
    ("small-tc-1row", SMALL_BF16, 1, 0.0, M.MOE_FFN_TCGEN05, None),
    ("small-tc", SMALL_BF16, 37, 1.0, M.MOE_FFN_TCGEN05, None),
    ("qwen-tc", W.QWEN3_30B_A3B, 65, 1.0, M.MOE_FFN_TCGEN05, 24),
    ("qwen-tc-skewed", W.QWEN3_30B_A3B, 65, 3.0, M.MOE_FFN_TCGEN05, 24),
    ("qwen-tc-4160rows", W.QWEN3_30B_A3B, 4160, 0.8, M.MOE_FFN_TCGEN05, 16),
    ("qwen-tc-600rows-hot", W.QWEN3_30B_A3B, 600, 2.0, M.MOE_FFN_TCGEN05, 16),
    ("qwen-tc-260rows", W.QWEN3_30B_A3B, 260, 1.0, M.MOE_FFN_TCGEN05, 32),
    ("gptoss-tc", GPTOSS32, 65, 0.7, M.MOE_FFN_TCGEN05, 24),
    ("e256-4000rows", W.LayerShape(d=256, E=256, k=4, f=128, dtype="bf16"), 4000, 0.5,
     M.MOE_FFN_TCGEN05, 24),
]


@pytest.mark.parametrize("case", EXPERT_CASES, ids=[c[0] for c in EXPERT_CASES])
def test_expert_forward(case):
    _, shape, R, skew, path, rows = case
    L = _desc(shape)
    wg, wu, wd = _weights(shape, 41)
    chain = np.arange(-1, R - 1, dtype=np.int32)
    x = W.hidden_states(42, chain, shape.d, shape.torch_dtype)
    idx = W.random_assignments(43, R, shape.E, shape.k, skew)
    gates = W.random_gates(44, R, shape.k)
    y = torch.empty(R, shape.d, dtype=shape.torch_dtype, device=DEV)
    ws = M.workspace(L, 1, R)
    M.moe_expert_forward(L, x.to(DEV), wg, wu, wd, None, torch.from_numpy(idx).to(DEV),
                         torch.from_numpy(gates).to(DEV), y, ws, M.run_opts(path))
    _sync()
    assert M.moe_workspace_check(ws) == 0
    sample = np.arange(R) if rows is None else np.random.default_rng(1).choice(R, rows, False)
    ref = O.moe_combine(x, wg.cpu(), wu.cpu(), wd.cpu(), idx, gates.astype(np.float64),
                        rows=sample.tolist())
    _assert_close_rows(y.float().cpu().numpy()[sample], ref, shape)


@pytest.mark.parametrize("path", [M.MOE_FFN_SIMT, M.MOE_FFN_TCGEN05])
def test_expert_forward_at_the_largest_width(path):
    """d = f = 6144, the largest hidden and SwiGLU width the layer accepts (the CUDA-core
    kernel stages 8 token rows of 6144 fp32 values in shared memory; the tensor-core kernel
    streams 96 k-chunks per unit), 4 experts, top-2, ragged 9 rows; sampled rows against
    the oracle."""
    shape = W.LayerShape(d=6144, E=4, k=2, f=6144, dtype="bf16")
    L = _desc(shape)
    R = 9
    wg, wu, wd = _weights(shape, 91)
    x = W.hidden_states(92, np.arange(-1, R - 1, dtype=np.int32), shape.d, torch.bfloat16)
    idx = W.random_assignments(93, R, shape.E, shape.k, 0.5)
    gates = W.random_gates(94, R, shape.k)
    y = torch.empty(R, shape.d, dtype=torch.bfloat16, device=DEV)
    ws = M.workspace(L, 1, R)
    M.moe_expert_forward(L, x.to(DEV), wg, wu, wd, None, torch.from_numpy(idx).to(DEV),
                         torch.from_numpy(gates).to(DEV), y, ws, M.run_opts(path))
    _sync()
    assert M.moe_workspace_check(ws) == 0
    rows = [0, 4, 8]
    ref = O.moe_combine(x, wg.cpu(), wu.cpu(), wd.cpu(), idx, gates.astype(np.float64),
                        rows=rows)
    _assert_close_rows(y.float().cpu().numpy()[rows], ref, shape)


def _assignments_with_counts(counts, R, k):
    """int32 [R, k] routing in which expert e takes exactly counts[e] assignments (sum =
    R * k, no count above R / 2 when k = 2), every row's experts distinct: the sorted list
    of expert ids, row r taking entries r, r + R, ... of it."""
    flat = np.repeat(np.arange(len(counts), dtype=np.int32), counts)
    assert flat.size == R * k
    idx = np.stack([flat[j * R:(j + 1) * R] for j in range(k)], axis=1)
    assert all(len(set(row)) == k for row in idx.tolist())
    return np.ascontiguousarray(idx)


@pytest.mark.parametrize("counts", [
    [256, 257, 384, 385, 700, 17, 0, 201],     # one tile of 256, equal tiles from 257 on
    [16, 300, 1000, 384, 96, 368, 0, 36],      # a hot expert in four tiles
    [256, 1, 512, 1, 255, 1, 510, 0]])         # full tiles next to one-token tiles
@pytest.mark.parametrize("max_ctas", [0, 8])
def test_expert_forward_exact_expert_loads(counts, max_ctas):
    """Experts with exactly the given numbers of tokens on the tensor-core path, around the
    256-token row-tile limit: a full 256-token tile (N = 256), experts of 257 tokens and
    more in near-equal tiles that share their weight loads, a hot expert in four tiles,
    one-token tiles, an expert with no tokens; every row against the oracle, on every SM
    and on 8 CTAs, where these few units take weight-tile pairs (one accumulator per tile of
    the pair over tiles taller than 128 tokens)."""
    shape = W.LayerShape(d=256, E=8, k=2, f=192, dtype="bf16")
    R = sum(counts) // 2
    L = _desc(shape)
    wg, wu, wd = _weights(shape, 51)
    x = W.hidden_states(52, np.arange(-1, R - 1, dtype=np.int32), shape.d, torch.bfloat16)
    idx = _assignments_with_counts(counts, R, 2)
    gates = W.random_gates(54, R, 2)
    y = torch.full((R, shape.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = M.workspace(L, 1, R)
    M.moe_expert_forward(L, x.to(DEV), wg, wu, wd, None, torch.from_numpy(idx).to(DEV),
                         torch.from_numpy(gates).to(DEV), y, ws,
                         M.run_opts(M.MOE_FFN_TCGEN05, ffn_max_ctas=max_ctas))
    _sync()
    assert M.moe_workspace_check(ws) == 0
    ref = O.moe_combine(x, wg.cpu(), wu.cpu(), wd.cpu(), idx, gates.astype(np.float64))
    _assert_close_rows(y.float().cpu().numpy(), ref, shape)


@pytest.mark.parametrize("counts,d,f", [
    ([128, 120, 33, 1, 0, 96, 65, 113], 320, 192),  # tallest tile 128: pairs fill 512 columns
    ([32, 32, 17, 31, 16, 32, 30, 10], 320, 192),   # tallest tile 32: the smallest paired
    ([128, 120, 33, 1, 0, 96, 65, 113], 256, 128),  # weight tiles in even counts
    ([31, 31, 17, 31, 16, 31, 30, 13], 320, 192),   # tallest tile 31 (32 rows): paired
    ([129, 128, 200, 230, 1, 0, 150, 200], 320, 192)])  # no expert past 256: 128-token split
@pytest.mark.parametrize("max_ctas", [0, 8])
def test_expert_forward_weight_tile_pairs(counts, d, f, max_ctas):
    """Row tiles of 32 to 128 tokens, where a unit of the tensor-core kernel takes two weight
    tiles that share the token rows: an odd number of weight tiles per phase (f = 192: 3
    tiles of 64 gate/up rows; d = 320: 3 tiles of 128 down rows, the last one 64 rows), so
    the last unit of each row tile holds one tile; the tallest tile at 128 tokens, where
    the second accumulator's second half ends at the last TMEM column; experts of 129-256
    tokens in two tiles of at most 128 (an expert of 128 tokens keeps one tile of 128,
    taller than the 65 + 64 of its neighbour of 129); every row against the oracle. On 8
    CTAs the kernel pairs at any number of units; on every SM these few units stay single
    (both must agree with the oracle)."""
    shape = W.LayerShape(d=d, E=8, k=2, f=f, dtype="bf16")
    R = sum(counts) // 2
    L = _desc(shape)
    wg, wu, wd = _weights(shape, 55)
    x = W.hidden_states(56, np.arange(-1, R - 1, dtype=np.int32), shape.d, torch.bfloat16)
    idx = _assignments_with_counts(counts, R, 2)
    gates = W.random_gates(57, R, 2)
    y = torch.full((R, shape.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = M.workspace(L, 1, R)
    M.moe_expert_forward(L, x.to(DEV), wg, wu, wd, None, torch.from_numpy(idx).to(DEV),
                         torch.from_numpy(gates).to(DEV), y, ws,
                         M.run_opts(M.MOE_FFN_TCGEN05, ffn_max_ctas=max_ctas))
    _sync()
    assert M.moe_workspace_check(ws) == 0
    ref = O.moe_combine(x, wg.cpu(), wu.cpu(), wd.cpu(), idx, gates.astype(np.float64))
    _assert_close_rows(y.float().cpu().numpy(), ref, shape)


@pytest.mark.parametrize("seed,max_ctas", [(0, 0), (15, 0), (0, 16)])
def test_one_tree_of_256_nodes_with_hot_experts(seed, max_ctas):
    """One tree of 256 nodes over 8 experts, top-2 (the selection cluster's own permute step
    builds the row tiles): experts of 140-173 tokens split in two near-equal tiles of at most
    128 tokens, which the tensor-core kernel on 16 CTAs runs in weight-tile pairs; counts,
    offsets and every row of y against the oracle."""
    shape = W.LayerShape(d=256, E=8, k=2, f=192, dtype="bf16")
    N, E, k = 256, 8, 2
    parent, depth = _tree_of(N, 70000 + seed)
    x = W.hidden_states(71000 + seed, parent, shape.d, torch.bfloat16)
    wr = W.router_weight(72000 + seed, shape, std=0.3)
    wg, wu, wd = _weights(shape, 73)
    L = _desc(shape)
    P = M.select_params(M.MOE_ROUTE_NATURAL, W.C_EAGLE)
    out = dict(logits=torch.empty(N, E, device=DEV),
               topk_idx=torch.empty(N, k, dtype=torch.int32, device=DEV),
               gates=torch.empty(N, k, device=DEV),
               eligible=torch.empty(1, E, dtype=torch.uint8, device=DEV),
               info=torch.empty(1, NF, dtype=torch.int32, device=DEV),
               counts=torch.empty(E, dtype=torch.int32, device=DEV),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV))
    y = torch.full((N, shape.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = M.workspace(L, 1, N)
    M.moe_tree_forward(L, P, x.to(DEV), wr.to(DEV), wg, wu, wd, None,
                       torch.from_numpy(depth.astype(np.int32)).to(DEV), 1, N, None, y, ws,
                       M.tree_outputs(**out),
                       M.run_opts(M.MOE_FFN_TCGEN05, ffn_max_ctas=max_ctas))
    _sync()
    assert M.moe_workspace_check(ws) == 0
    got = {key: v.cpu().numpy() for key, v in out.items()}
    assert 128 < got["counts"].max() <= 256  # the case this test is for
    rc, ro, _ = O.permute(got["topk_idx"], E)
    np.testing.assert_array_equal(got["counts"], rc)
    np.testing.assert_array_equal(got["offsets"], ro)
    ref = O.moe_combine(x, wg.cpu(), wu.cpu(), wd.cpu(), got["topk_idx"], got["gates"])
    _assert_close_rows(y.float().cpu().numpy(), ref, shape)


def test_selection_cluster_at_its_largest_tree():
    """256 nodes (the largest tree the 8-CTA cluster takes), E = 256, k = 16: the launch
    with the most shared memory (logit rows, fp32 and fp64 demand terms of 32 nodes per
    CTA); AcceptMoE with pruning against the fp64 oracle, one tree exact per tree."""
    shape = W.LayerShape(d=64, E=256, k=16, f=64, dtype="fp32")
    N = 256
    parent, depth = _tree_of(N, 256)
    logits = W.synthetic_logits(257, parent[None], shape.E, 3.0)
    res = W.residency_mask(9, shape.E, 96)
    kw = dict(mode=O.ACCEPT, prune=True, budget=8, min_set=24, resident=res, c=W.C_EAGLE)
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE, prune=True, reroute_budget=8,
                        min_set=24)
    gidx, gg, ge, gi = _select_gpu(shape, P, logits, depth[None], 1, N, res)
    assert _check_selection(shape, kw, logits, depth[None], gidx, gg, ge, gi, N, 1) == 0


@pytest.mark.parametrize("shape,R,skew", [(SMALL_BF16, 65, 1.0), (W.QWEN3_30B_A3B, 65, 1.0),
                                          (W.QWEN3_30B_A3B, 520, 2.0), (GPTOSS32, 33, 0.5)])
def test_tcgen05_matches_simt(shape, R, skew):
    """The tensor-core and CUDA-core expert kernels agree on the same inputs."""
    L = _desc(shape)
    wg, wu, wd = _weights(shape, 61)
    x = W.hidden_states(62, np.arange(-1, R - 1, dtype=np.int32), shape.d, shape.torch_dtype)
    ti = torch.from_numpy(W.random_assignments(63, R, shape.E, shape.k, skew)).to(DEV)
    tg = torch.from_numpy(W.random_gates(64, R, shape.k)).to(DEV)
    ys = []
    for path in (M.MOE_FFN_SIMT, M.MOE_FFN_TCGEN05):
        y = torch.empty(R, shape.d, dtype=shape.torch_dtype, device=DEV)
        ws = M.workspace(L, 1, R)
        M.moe_expert_forward(L, x.to(DEV), wg, wu, wd, None, ti, tg, y, ws, M.run_opts(path))
        _sync()
        assert M.moe_workspace_check(ws) == 0
        ys.append(y.float().cpu().numpy())
    ref = ys[0].astype(np.float64)
    assert np.abs(ys[1] - ref).max() <= 2e-2 * np.abs(ref).max()


def test_tcgen05_slot_pool_larger_than_E():
    """Experts addressed through a slot map into a pool of S > E slots (the offload
    layout): same result as the plain [E] layout."""
    shape = SMALL_BF16
    S = 24
    wg, wu, wd = _weights(shape, 71)
    slot = np.random.default_rng(5).choice(S, shape.E, replace=False).astype(np.int32)
    pg = torch.zeros(S, shape.f, shape.d, dtype=torch.bfloat16, device=DEV)
    pu, pd = torch.zeros_like(pg), torch.zeros(S, shape.d, shape.f, dtype=torch.bfloat16,
                                               device=DEV)
    ts = torch.from_numpy(slot).long().to(DEV)
    pg[ts], pu[ts], pd[ts] = wg, wu, wd
    R = 40
    x = W.hidden_states(72, np.arange(-1, R - 1, dtype=np.int32), shape.d, torch.bfloat16).to(DEV)
    ti = torch.from_numpy(W.random_assignments(73, R, shape.E, shape.k)).to(DEV)
    tg = torch.from_numpy(W.random_gates(74, R, shape.k)).to(DEV)
    y0 = torch.empty(R, shape.d, dtype=torch.bfloat16, device=DEV)
    y1 = torch.empty_like(y0)
    L = _desc(shape)
    Ls = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16", slots=S)
    ws = M.workspace(L, 1, R)
    M.moe_expert_forward(L, x, wg, wu, wd, None, ti, tg, y0, ws, M.run_opts(M.MOE_FFN_TCGEN05))
    M.moe_expert_forward(Ls, x, pg, pu, pd, torch.from_numpy(slot).to(DEV), ti, tg, y1, ws,
                         M.run_opts(M.MOE_FFN_TCGEN05))
    _sync()
    assert M.moe_workspace_check(ws) == 0
    assert torch.equal(y0, y1)


def test_expert_forward_slot_map():
    """Experts addressed through a slot map (the offload layout) give the same y."""
    shape = W.TINY
    L = _desc(shape)
    wg, wu, wd = _weights(shape, 51)
    perm = np.random.default_rng(2).permutation(shape.E).astype(np.int32)  # expert -> slot
    inv = np.argsort(perm)
    sg, su, sd = wg[torch.from_numpy(inv).to(DEV)], wu[torch.from_numpy(inv).to(DEV)], \
        wd[torch.from_numpy(inv).to(DEV)]
    R = 17
    x = W.hidden_states(52, np.arange(-1, R - 1, dtype=np.int32), shape.d, torch.float32)
    idx = W.random_assignments(53, R, shape.E, shape.k)
    gates = W.random_gates(54, R, shape.k)
    y0 = torch.empty(R, shape.d, device=DEV)
    y1 = torch.empty(R, shape.d, device=DEV)
    ws = M.workspace(L, 1, R)
    ti, tg = torch.from_numpy(idx).to(DEV), torch.from_numpy(gates).to(DEV)
    M.moe_expert_forward(L, x.to(DEV), wg, wu, wd, None, ti, tg, y0, ws)
    M.moe_expert_forward(L, x.to(DEV), sg.contiguous(), su.contiguous(), sd.contiguous(),
                         torch.from_numpy(perm).to(DEV), ti, tg, y1, ws)
    _sync()
    assert torch.equal(y0, y1)


# -------------------------------------------------------------- whole layer

FORWARD_CASES = [
    # (id, shape, B, tree kind, router std, mode, sampled rows or None)
    ("cfg0-nat", W.TINY, 1, "tiny", 0.02, M.MOE_ROUTE_NATURAL, None),
    ("cfg0-acc", W.TINY, 1, "tiny", 0.02, M.MOE_ROUTE_ACCEPT, None),
    ("cfg0-acc-peaked", W.TINY, 1, "tiny", 0.3, M.MOE_ROUTE_ACCEPT, None),
    ("cfg1-nat", W.QWEN3_30B_A3B, 1, "eagle", 0.02, M.MOE_ROUTE_NATURAL, 12),
    ("cfg1-acc", W.QWEN3_30B_A3B, 1, "eagle", 0.02, M.MOE_ROUTE_ACCEPT, 12),
    ("cfg1-acc-peaked", W.QWEN3_30B_A3B, 1, "eagle", 0.1, M.MOE_ROUTE_ACCEPT, 12),
    ("cfg4-b4-acc-peaked", W.QWEN3_30B_A3B, 4, "eagle", 0.1, M.MOE_ROUTE_ACCEPT, 12),
    ("cfg4-b16-nat", W.QWEN3_30B_A3B, 16, "eagle", 0.02, M.MOE_ROUTE_NATURAL, 12),
    ("cfg4-b64-acc-peaked", W.QWEN3_30B_A3B, 64, "eagle", 0.1, M.MOE_ROUTE_ACCEPT, 8),
    ("gptoss-acc-peaked", W.GPT_OSS_120B, 1, "eagle", 0.1, M.MOE_ROUTE_ACCEPT, 8),
]


def _run_forward(shape, B, kind, std, mode, seed, path=M.MOE_FFN_AUTO, prune=None):
    c = W.C_TINY if kind == "tiny" else W.C_EAGLE
    parent, depth = W.tree_block(seed, B, kind)
    N = parent.shape[1]
    R = B * N
    x = W.hidden_states(seed + 1, parent, shape.d, shape.torch_dtype)
    wr = W.router_weight(seed + 2, shape, std=std)
    wg, wu, wd = _weights(shape, seed + 3)
    L = _desc(shape)
    P = M.select_params(mode, c)
    out = dict(logits=torch.empty(R, shape.E, device=DEV),
               topk_idx=torch.empty(R, shape.k, dtype=torch.int32, device=DEV),
               gates=torch.empty(R, shape.k, device=DEV),
               eligible=torch.empty(B, shape.E, dtype=torch.uint8, device=DEV),
               info=torch.empty(B, NF, dtype=torch.int32, device=DEV),
               counts=torch.empty(shape.E, dtype=torch.int32, device=DEV),
               offsets=torch.empty(shape.E + 1, dtype=torch.int32, device=DEV),
               perm=torch.empty(R * shape.k, dtype=torch.int32, device=DEV))
    y = torch.empty(R, shape.d, dtype=shape.torch_dtype, device=DEV)
    ws = M.workspace(L, B, N)
    dp = torch.from_numpy(depth.reshape(-1).copy()).to(DEV)
    M.moe_tree_forward(L, P, x.to(DEV), wr.to(DEV), wg, wu, wd, None, dp, B, N, None, y, ws,
                       M.tree_outputs(**out), M.run_opts(path))
    _sync()
    assert M.moe_workspace_check(ws) == 0
    got = {k: v.cpu().numpy() for k, v in out.items()}
    got["y"] = y.float().cpu().numpy()
    return dict(x=x, wr=wr, wg=wg, wu=wu, wd=wd, depth=depth, c=c, N=N, got=got)


@pytest.mark.parametrize("case", FORWARD_CASES, ids=[c[0] for c in FORWARD_CASES])
def test_tree_forward_against_oracle(case):
    """The whole layer. The router's logits are compared with the oracle's (its own fp64
    matmul); every later step is compared with the oracle fed the device's fp32 logits,
    exactly (per tree, fp64 ties excused as in the selection tests); the layer output on
    sampled rows is compared with the oracle's experts and combine on those choices. The
    oracle's routing from its own logits must also agree on nearly every row."""
    _, shape, B, kind, std, mode, rows = case
    run = _run_forward(shape, B, kind, std, mode, seed=300 + B)
    got, N = run["got"], run["N"]
    R = B * N
    omode = {M.MOE_ROUTE_NATURAL: O.NATURAL, M.MOE_ROUTE_ACCEPT: O.ACCEPT}[mode]
    sample = list(range(R)) if rows is None else \
        sorted(np.random.default_rng(3).choice(R, rows, replace=False).tolist())
    # 1. router logits against the oracle's own
    ref_l = O.router(run["x"], run["wr"])
    scale = np.abs(ref_l).max(axis=1, keepdims=True)
    assert (np.abs(got["logits"] - ref_l) <= 1e-4 * scale).all()
    # 2. selection, permute and counters from the device's logits, tree by tree
    depth = run["depth"]
    kw = dict(mode=omode, c=run["c"])
    tied = _check_selection(shape, kw, got["logits"], depth, got["topk_idx"], got["gates"],
                            got["eligible"], got["info"], N, B)
    assert tied == 0
    rc, ro, rp = O.permute(got["topk_idx"], shape.E)
    np.testing.assert_array_equal(got["counts"], rc)
    np.testing.assert_array_equal(got["offsets"], ro)
    np.testing.assert_array_equal(got["perm"], rp)
    sel = O.select_block(got["logits"], depth, shape.k, run["c"], mode=omode)
    np.testing.assert_array_equal(got["topk_idx"], sel["idx"])
    # 3. the layer output on sampled rows: the oracle's experts and combine
    y_ref = O.moe_combine(run["x"], run["wg"].cpu(), run["wu"].cpu(), run["wd"].cpu(),
                          sel["idx"], sel["gates"], rows=sample)
    _assert_close_rows(got["y"][sample], y_ref, shape)
    # 4. the oracle end to end from its own logits: the same routing on nearly every row
    # (rows may differ only where the two logit computations straddle a near-tie)
    own = O.select_block(ref_l.astype(np.float32), depth, shape.k, run["c"], mode=omode)
    same = (np.sort(own["idx"], axis=1) == np.sort(got["topk_idx"], axis=1)).all(axis=1)
    assert same.mean() >= 0.98, same.mean()
    # invariants that hold at any size
    for b in range(B):
        S = set(np.flatnonzero(got["eligible"][b]).tolist())
        chosen = set(np.unique(got["topk_idx"][b * N:(b + 1) * N]).tolist())
        assert chosen <= S and len(S) >= shape.k
        assert got["info"][b, 1] <= got["info"][b, 0]


def test_tree_forward_is_deterministic():
    a = _run_forward(W.QWEN3_30B_A3B, 1, "eagle", 0.1, M.MOE_ROUTE_ACCEPT, seed=77)
    b = _run_forward(W.QWEN3_30B_A3B, 1, "eagle", 0.1, M.MOE_ROUTE_ACCEPT, seed=77)
    for k in a["got"]:
        np.testing.assert_array_equal(a["got"][k], b["got"][k])


def test_residual_chain_of_layers_against_oracle():
    """Three Qwen3-shaped layers in a residual chain, x <- x + MoE_l(x) with x stored in
    bf16 between layers (the 48-layer stack's step). The oracle runs the chain itself from
    the same seeded inputs, rounding each layer's x to bf16 as the stored dtype requires."""
    shape = W.QWEN3_30B_A3B
    t = W.eagle_tree(900)
    N = t.N
    x0 = W.hidden_states(901, t.parent, shape.d, torch.bfloat16)
    L = _desc(shape)
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    layers = [(W.router_weight(910 + l, shape, std=0.1, device=DEV),) + _weights(shape, 920 + l)
              for l in range(3)]
    x = x0.to(DEV).clone()
    dep = torch.from_numpy(t.depth.copy()).to(DEV)
    ws = M.workspace(L, 1, N)
    idx = torch.empty(N, shape.k, dtype=torch.int32, device=DEV)
    got_idx = []
    for wr, wg, wu, wd in layers:
        M.moe_tree_forward(L, P, x, wr, wg, wu, wd, None, dep, 1, N, None, x, ws,
                           M.tree_outputs(topk_idx=idx), M.run_opts(residual=True))
        torch.cuda.synchronize()
        got_idx.append(idx.cpu().numpy().copy())
    xo = x0
    for l, (wr, wg, wu, wd) in enumerate(layers):
        ref = O.forward(xo, wr.cpu(), wg.cpu(), wu.cpu(), wd.cpu(), t.depth, shape.k, W.C_EAGLE,
                        mode=O.ACCEPT)
        # identical inputs for the first layer, inputs that differ by the bf16 rounding of
        # the previous layer's output afterwards: the routing agrees on nearly every row
        same = sum(set(got_idx[l][r].tolist()) == set(ref["idx"][r].tolist())
                   for r in range(N))
        assert same >= (0.98 if l == 0 else 0.9) * N
        xo = (xo.double() + torch.from_numpy(ref["y"])).to(torch.bfloat16)
    ref_x = xo.double().numpy()
    got = x.double().cpu().numpy()
    assert np.abs(got - ref_x).max() <= 2e-2 * np.abs(ref_x).max()


# ------------------------------------------------- cost-aware draft selection

def _sel_tree_from_oracle(cand, sel):
    pos = {int(v): i for i, v in enumerate(sel)}
    par = np.array([-1] + [pos[int(cand.parent[v])] for v in sel[1:]], np.int32)
    return par, cand.depth[sel]


@pytest.mark.parametrize("lam", [0.0, 0.2, 1.0])
def test_draft_select_bit_exact(lam):
    shape = W.QWEN3_30B_A3B
    L = _desc(shape)
    cand = W.eagle_candidates(77)
    logits = W.synthetic_logits(78, cand.parent, shape.E, 2.0)
    fp, _ = O.topk(logits, shape.k)
    x = W.hidden_states(79, cand.parent, shape.d, torch.bfloat16)
    gamma = 65
    sel = torch.empty(gamma, dtype=torch.int32, device=DEV)
    spar, sdep = torch.empty_like(sel), torch.empty_like(sel)
    x_sel = torch.empty(gamma, shape.d, dtype=torch.bfloat16, device=DEV)
    nu = torch.empty(1, dtype=torch.int32, device=DEV)
    td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    M.moe_draft_select(L, td(cand.parent), td(cand.depth), td(cand.logp), td(fp), lam, gamma,
                       sel, spar, sdep, x.to(DEV), x_sel, nu)
    _sync()
    ref_sel, ref_u = O.draft_select(cand.parent, cand.logp, fp, shape.E, lam, gamma)
    np.testing.assert_array_equal(sel.cpu().numpy(), ref_sel)
    rp, rd = _sel_tree_from_oracle(cand, ref_sel)
    np.testing.assert_array_equal(spar.cpu().numpy(), rp)
    np.testing.assert_array_equal(sdep.cpu().numpy(), rd)
    assert int(nu.item()) == ref_u
    assert torch.equal(x_sel.cpu(), x[torch.from_numpy(ref_sel).long()])


@pytest.mark.parametrize("steps,topk,E,k,lam,junk", [
    (9, 12, 256, 16, 0.05, False),   # C = 1165: two candidates per thread, 8-word bit sets
    (8, 20, 128, 8, 0.3, False),     # C = 2821: four candidates per thread
    (3, 6, 64, 4, 0.5, True),        # repeated and out-of-range footprint ids
])
def test_draft_select_large_and_junk_footprints(steps, topk, E, k, lam, junk):
    cand = W.eagle_candidates(90 + steps, steps=steps, topk=topk)
    C = cand.C
    rng = np.random.default_rng(91 + steps)
    if junk:
        fp = rng.integers(-3, E + 3, size=(C, k)).astype(np.int32)
        fp[:, 1] = fp[:, 0]  # every footprint lists one id twice
    else:
        fp = np.stack([rng.choice(E, size=k, replace=False) for _ in range(C)]).astype(np.int32)
    L = M.layer_desc(256, E, k, 128, "bf16")
    gamma = min(200, C)
    sel = torch.empty(gamma, dtype=torch.int32, device=DEV)
    spar, sdep = torch.empty_like(sel), torch.empty_like(sel)
    nu = torch.empty(1, dtype=torch.int32, device=DEV)
    td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    M.moe_draft_select(L, td(cand.parent), td(cand.depth), td(cand.logp), td(fp), lam, gamma,
                       sel, spar, sdep, n_union=nu)
    _sync()
    ref_sel, ref_u = O.draft_select(cand.parent, cand.logp, fp, E, lam, gamma)
    np.testing.assert_array_equal(sel.cpu().numpy(), ref_sel)
    rp, rd = _sel_tree_from_oracle(cand, ref_sel)
    np.testing.assert_array_equal(spar.cpu().numpy(), rp)
    np.testing.assert_array_equal(sdep.cpu().numpy(), rd)
    assert int(nu.item()) == ref_u


def test_draft_select_fewer_candidates_than_gamma():
    parent = np.array([-1, 0, 0, 1, 7], np.int32)  # node 4's parent is out of range
    depth = np.array([0, 1, 1, 2, 3], np.int32)
    logp = np.array([0.0, -0.5, -0.7, -0.9, -0.1], np.float32)
    fp = np.array([[0, 1], [2, 3], [0, 1], [2, 4], [5, 6]], np.int32)
    L = M.layer_desc(256, 8, 2, 128, "bf16")
    gamma = 8
    sel = torch.full((gamma,), 99, dtype=torch.int32, device=DEV)
    spar, sdep = torch.full_like(sel, 99), torch.full_like(sel, 99)
    nu = torch.empty(1, dtype=torch.int32, device=DEV)
    td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    M.moe_draft_select(L, td(parent), td(depth), td(logp), td(fp), 0.1, gamma, sel, spar, sdep,
                       n_union=nu)
    _sync()
    ref_sel, ref_u = O.draft_select(parent, logp, fp, 8, 0.1, gamma)
    assert ref_sel.tolist() == [0, 1, 2, 3]
    assert sel.cpu().tolist() == [0, 1, 2, 3, -1, -1, -1, -1]
    assert spar.cpu().tolist() == [-1, 0, 0, 1, -1, -1, -1, -1]
    assert sdep.cpu().tolist() == [0, 1, 1, 2, -1, -1, -1, -1]
    assert int(nu.item()) == ref_u == 5


def test_draft_select_then_verify_against_oracle():
    """The whole cost-aware pipeline on the device: router over every candidate, the
    natural top-k as the predicted footprint, the selection, and verification of the
    chosen tree (natural routing); the oracle runs the same steps from the same inputs."""
    shape = W.QWEN3_30B_A3B
    L = _desc(shape)
    cand = W.eagle_candidates(81)
    C = cand.C
    x = W.hidden_states(82, cand.parent, shape.d, torch.bfloat16)
    wr = W.router_weight(83, shape, std=0.1)
    wg, wu, wd = _weights(shape, 84)
    td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    logits = torch.empty(C, shape.E, device=DEV)
    M.moe_router_logits(L, x.to(DEV), wr.to(DEV), logits)
    fp = torch.empty(C, shape.k, dtype=torch.int32, device=DEV)
    g = torch.empty(C, shape.k, device=DEV)
    M.moe_tree_select(L, M.select_params(M.MOE_ROUTE_NATURAL, [1.0]), logits, td(cand.depth), 1,
                      C, None, fp, g)
    gamma, lam = 65, 0.3
    sel = torch.empty(gamma, dtype=torch.int32, device=DEV)
    spar, sdep = torch.empty_like(sel), torch.empty_like(sel)
    x_sel = torch.empty(gamma, shape.d, dtype=torch.bfloat16, device=DEV)
    M.moe_draft_select(L, td(cand.parent), td(cand.depth), td(cand.logp), fp, lam, gamma, sel,
                       spar, sdep, x.to(DEV), x_sel)
    y = torch.empty_like(x_sel)
    ws = M.workspace(L, 1, gamma)
    idx = torch.empty(gamma, shape.k, dtype=torch.int32, device=DEV)
    M.moe_tree_forward(L, M.select_params(M.MOE_ROUTE_NATURAL, [1.0]), x_sel, wr.to(DEV), wg, wu,
                       wd, None, sdep, 1, gamma, None, y, ws, M.tree_outputs(topk_idx=idx))
    _sync()
    l32 = O.router(x, wr).astype(np.float32)
    rfp, _ = O.topk(l32, shape.k)
    srt = -np.sort(-l32, axis=1)
    boundary = srt[:, shape.k - 1] - srt[:, shape.k]  # k-th vs (k+1)-th logit
    tied = boundary < 1e-5 * np.abs(srt[:, 0])
    gfp = fp.cpu().numpy()
    same = [set(gfp[r].tolist()) == set(rfp[r].tolist()) for r in range(C)]
    assert all(same[r] for r in range(C) if not tied[r])
    if not all(same):
        pytest.skip("a footprint decided by an fp32 tie: both selections are valid")
    ref_sel, _ = O.draft_select(cand.parent, cand.logp, rfp, shape.E, lam, gamma)
    np.testing.assert_array_equal(sel.cpu().numpy(), ref_sel)
    xs = x[torch.from_numpy(ref_sel).long()]
    rows = list(range(0, gamma, 6))
    ref = O.forward(xs, wr, wg.cpu(), wu.cpu(), wd.cpu(), cand.depth[ref_sel], shape.k, [1.0],
                    rows=rows, mode=O.NATURAL)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"])
    _assert_close_rows(y.float().cpu().numpy()[rows], ref["y"], shape)


E256_BF16 = W.LayerShape(d=256, E=256, k=8, f=128, dtype="bf16")


@pytest.mark.parametrize("shape,draft_tokens,mode", [
    (E256_BF16, 64, M.MOE_ROUTE_ACCEPT),           # one tree: selection cluster permutes, 8 logits/lane
    (E256_BF16, 64, M.MOE_ROUTE_NATURAL),          # one tree: natural cluster permutes
    (W.QWEN3_30B_A3B, 299, M.MOE_ROUTE_ACCEPT),    # 300 nodes: one-CTA selection + permute kernel
    (W.QWEN3_30B_A3B, 299, M.MOE_ROUTE_NATURAL),   # 300 nodes: permute kernel
], ids=["e256-acc", "e256-nat", "n300-acc", "n300-nat"])
def test_tree_forward_permute_outputs(shape, draft_tokens, mode):
    """The layer's permute outputs, whichever kernel produced them (the selection launch for
    a block of one tree of up to 256 nodes, else the permute kernel), equal the oracle's
    counting sort of the layer's own expert choices, and the standalone permute kernel's;
    the layer output matches the oracle on sampled rows."""
    t = W.eagle_tree(4242, draft_tokens=draft_tokens)
    N = t.N
    x = W.hidden_states(4243, t.parent, shape.d, shape.torch_dtype)
    wr = W.router_weight(4244, shape, std=0.1)
    wg, wu, wd = _weights(shape, 4245)
    L = _desc(shape)
    P = M.select_params(mode, W.C_EAGLE)
    idx = torch.empty(N, shape.k, dtype=torch.int32, device=DEV)
    counts = torch.empty(shape.E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(shape.E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(N * shape.k, dtype=torch.int32, device=DEV)
    y = torch.empty(N, shape.d, dtype=shape.torch_dtype, device=DEV)
    ws = M.workspace(L, 1, N)
    dp = torch.from_numpy(t.depth.copy()).to(DEV)
    M.moe_tree_forward(L, P, x.to(DEV), wr.to(DEV), wg, wu, wd, None, dp, 1, N, None, y, ws,
                       M.tree_outputs(topk_idx=idx, counts=counts, offsets=offsets, perm=perm))
    _sync()
    assert M.moe_workspace_check(ws) == 0
    got_idx = idx.cpu().numpy()
    rc, ro, rp = O.permute(got_idx, shape.E)
    np.testing.assert_array_equal(counts.cpu().numpy(), rc)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
    np.testing.assert_array_equal(perm.cpu().numpy(), rp)
    # the standalone permute kernel on the same choices
    c2, o2, p2 = torch.empty_like(counts), torch.empty_like(offsets), torch.empty_like(perm)
    ws2 = M.workspace(L, 1, N)
    M.moe_expert_permute(L, idx, c2, o2, p2, ws2)
    _sync()
    np.testing.assert_array_equal(c2.cpu().numpy(), counts.cpu().numpy())
    np.testing.assert_array_equal(o2.cpu().numpy(), offsets.cpu().numpy())
    np.testing.assert_array_equal(p2.cpu().numpy(), perm.cpu().numpy())
    # the layer output on sampled rows, against the oracle's combine of the same choices
    rows = sorted(np.random.default_rng(5).choice(N, 6, replace=False).tolist())
    gates = torch.empty(N, shape.k, device=DEV)
    M.moe_tree_forward(L, P, x.to(DEV), wr.to(DEV), wg, wu, wd, None, dp, 1, N, None, y, ws,
                       M.tree_outputs(gates=gates))
    _sync()
    yr = O.moe_combine(x, wg.cpu(), wu.cpu(), wd.cpu(), got_idx, gates.cpu().numpy(), rows=rows)
    _assert_close_rows(y.float().cpu().numpy()[rows], yr, shape)


@pytest.mark.parametrize("E,k", [(128, 8), (256, 8), (64, 4), (100, 16)])
def test_topk_with_exact_ties(E, k):
    """Logits drawn from three values, so nearly every top-k round has tied candidates in
    several lanes: the choices are the natural top-k with ties to the lower expert id, both
    in the natural-routing kernel and in the selection cluster (fixed size E over all
    experts, so every expert is eligible and the restricted top-k is the natural one)."""
    shape = W.LayerShape(d=64, E=E, k=k, f=64, dtype="fp32")
    N = 65
    rng = np.random.default_rng(E + k)
    logits = rng.integers(0, 3, size=(N, E)).astype(np.float32)
    logits[7] = 1.0  # a row of all-equal logits: the k lowest ids
    ref, _ = O.topk(logits, k)
    np.testing.assert_array_equal(ref[7], np.arange(k))
    depth = np.minimum(np.arange(N), 5).astype(np.int32)
    for mode, kw in ((M.MOE_ROUTE_NATURAL, {}),
                     (M.MOE_ROUTE_FIXED_B, dict(fixed_B=E, pool_all=True))):
        P = M.select_params(mode, W.C_EAGLE, **kw)
        gidx, _, _, _ = _select_gpu(shape, P, logits, depth, 1, N)
        np.testing.assert_array_equal(gidx, ref)


@pytest.mark.parametrize("cap", [1, 64, 136])
def test_two_streams_with_capped_expert_kernel(cap):
    """Two one-tree blocks in flight on two streams, each with its own workspace and the
    tensor-core expert kernel capped at `cap` CTAs, give the same routing and y bit for bit
    as the same trees run one at a time with one CTA per SM."""
    shape = W.QWEN3_30B_A3B
    L = _desc(shape)
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    wr = W.router_weight(960, shape, std=0.1, device=DEV)
    wg, wu, wd = _weights(shape, 961)
    trees = [W.eagle_tree(962 + i) for i in range(6)]
    xs = [W.hidden_states(970 + i, t.parent, shape.d, torch.bfloat16).to(DEV)
          for i, t in enumerate(trees)]
    deps = [torch.from_numpy(t.depth.copy()).to(DEV) for t in trees]
    streams = [torch.cuda.current_stream(), torch.cuda.Stream()]
    wss = [M.workspace(L, 1, 65), M.workspace(L, 1, 65)]
    ys = [torch.empty(t.N, shape.d, dtype=torch.bfloat16, device=DEV) for t in trees]
    idx = [torch.empty(t.N, shape.k, dtype=torch.int32, device=DEV) for t in trees]
    opts = M.run_opts(M.MOE_FFN_TCGEN05, ffn_max_ctas=cap)
    streams[1].wait_stream(streams[0])
    for i, t in enumerate(trees):
        M.moe_tree_forward(L, P, xs[i], wr, wg, wu, wd, None, deps[i], 1, t.N, None, ys[i],
                           wss[i % 2], M.tree_outputs(topk_idx=idx[i]), opts, streams[i % 2])
    streams[0].wait_stream(streams[1])
    _sync()
    for w_ in wss:
        assert M.moe_workspace_check(w_) == 0
    ws = M.workspace(L, 1, 65)
    for i, t in enumerate(trees):
        y = torch.empty_like(ys[i])
        i2 = torch.empty_like(idx[i])
        M.moe_tree_forward(L, P, xs[i], wr, wg, wu, wd, None, deps[i], 1, t.N, None, y, ws,
                           M.tree_outputs(topk_idx=i2), M.run_opts(M.MOE_FFN_TCGEN05))
        _sync()
        assert torch.equal(i2, idx[i]), i
        assert torch.equal(y, ys[i]), i
