"""Pins for the CPU oracle: worked examples, closed forms, brute force, invariants.

Each check ties the oracle to something other than itself: values printed on the
pages (tests/golden), closed forms (MoESD notes section 5.3, softmax/entropy of
structured inputs), library routines (torch fp64 matmul, torch silu, scipy
softmax), and brute-force enumeration on tiny inputs.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax as sp_softmax

from expert_select_gb300 import workload as W
from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    out = []
    with open(os.path.join(GOLD, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


# ---------------------------------------------------------------- worked examples

def test_worked_example_a_union_counts_reuse():
    rows = _read("worked_example_a.txt")
    E = int(next(r[1] for r in rows if r[0] == "E"))
    k = int(next(r[1] for r in rows if r[0] == "k"))
    sets = [[int(v) for v in r[1:]] for r in rows if r[0] == "row"]
    idx, _ = O.topk(W.routing_from_sets(sets, E), k)
    for r, s in enumerate(sets):
        assert sorted(idx[r].tolist()) == sorted(s)
    counts, offsets, perm = O.permute(idx, E)
    union = int((counts > 0).sum())
    assert int(counts.sum()) == int(next(r[1] for r in rows if r[0] == "expect_assignments"))
    assert union == int(next(r[1] for r in rows if r[0] == "expect_union"))
    for r in rows:
        if r[0] == "expect_count":
            assert counts[int(r[1])] == int(r[2])
    reuse = 1.0 - union / float(idx.size)
    assert reuse == pytest.approx(float(next(r[1] for r in rows if r[0] == "expect_reuse")))
    # the natural-mode selection reports the same union
    sel = O.select_tree(W.routing_from_sets(sets, E), np.array([0, 1, 1, 1]), k, [1.0],
                        mode=O.NATURAL)
    assert sel["union_nat"] == union == sel["union_sel"]
    dis = [[int(v) for v in r[1:]] for r in rows if r[0] == "disjoint_row"]
    didx, _ = O.topk(W.routing_from_sets(dis, E), k)
    dc, _, _ = O.permute(didx, E)
    assert int((dc > 0).sum()) == int(next(r[1] for r in rows if r[0] == "expect_disjoint_union"))


def test_worked_example_b_tree_union():
    rows = _read("worked_example_b.txt")
    E = int(next(r[1] for r in rows if r[0] == "E"))
    k = int(next(r[1] for r in rows if r[0] == "k"))
    nodes = [r for r in rows if r[0] == "node"]
    sets = [[int(v) for v in r[3:]] for r in nodes]
    idx, _ = O.topk(W.routing_from_sets(sets, E), k)
    counts, _, _ = O.permute(idx, E)
    assert int((counts > 0).sum()) == int(next(r[1] for r in rows if r[0] == "expect_union"))
    for r in rows:
        if r[0] == "expect_count":
            assert counts[int(r[1])] == int(r[2])


# ------------------------------------------------------------------ closed forms

@pytest.mark.parametrize("E,K,t", [(16, 2, 4), (16, 2, 5), (16, 2, 9), (128, 8, 65), (128, 4, 65)])
def test_union_expectation_closed_form(E, K, t):
    """MoESD notes section 5.3: with every token choosing K of E experts uniformly,
    the expected number of distinct experts after t tokens is E[1-((E-K)/E)^t].
    i.i.d. Gaussian logits make each natural top-K a uniform K-subset."""
    trials = 3000 if E == 16 else 600
    rng = np.random.Generator(np.random.PCG64(1234 + E + K + t))
    logits = rng.standard_normal((trials * t, E)).astype(np.float32)
    unions = np.empty(trials)
    for i in range(trials):
        sel = O.select_tree(logits[i * t:(i + 1) * t], np.zeros(t, np.int32), K, [1.0],
                            mode=O.NATURAL)
        unions[i] = sel["union_nat"]
    expect = E * (1.0 - ((E - K) / E) ** t)
    se = unions.std(ddof=1) / math.sqrt(trials)
    assert abs(unions.mean() - expect) < 4.0 * se + 1e-9, (unions.mean(), expect, se)


def test_router_matches_torch_fp64():
    g = torch.Generator().manual_seed(7)
    for dt in (torch.float32, torch.bfloat16):
        x = torch.randn(7, 96, generator=g).to(dt)
        w = (torch.randn(12, 96, generator=g) * 0.05).to(dt)
        ref = (x.double() @ w.double().T).numpy()
        got = O.router(x, w)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_topk_brute_force_with_ties():
    rng = np.random.Generator(np.random.PCG64(5))
    for trial in range(50):
        E, k = int(rng.integers(3, 24)), None
        k = int(rng.integers(1, E + 1))
        # coarse values force ties; ties must go to the lower expert id
        l = np.round(rng.standard_normal((6, E)) * 2) .astype(np.float32)
        idx, _ = O.topk(l, k)
        for r in range(6):
            ref = sorted(range(E), key=lambda e: (-float(l[r, e]), e))[:k]
            assert idx[r].tolist() == ref


def _one_hot_logits(hot, E):
    """Rows whose softmax is exactly one-hot in fp64 (exp(-1000) underflows to 0)."""
    l = np.full((len(hot), E), -1000.0, dtype=np.float32)
    for r, e in enumerate(hot):
        l[r, e] = 0.0
    return l


def test_demand_one_hot_closed_form_and_depth_table():
    """One-hot routing makes D_e = sum of c(depth_n) over the nodes routed to e,
    and depths past the end of the commitment table use its last entry."""
    E, k = 12, 1
    c = [1.0, 0.5, 0.25]
    depth = np.array([0, 1, 1, 2, 3, 7, 2], dtype=np.int32)
    hot = [3, 5, 5, 3, 9, 9, 0]
    sel = O.select_tree(_one_hot_logits(hot, E), depth, k, c, mode=O.ACCEPT, pool_all=True)
    ct = [c[min(t, 2)] for t in depth]
    expect = np.zeros(E)
    for n, e in enumerate(hot):
        expect[e] += ct[n]
    np.testing.assert_array_equal(sel["D"], expect)
    q = expect[expect > 0] / expect.sum()
    rank = math.exp(-(q * np.log(q)).sum())
    assert sel["m"] == max(k, math.ceil(rank - 1e-12))


@pytest.mark.parametrize("j", [1, 3, 8, 13])
def test_uniform_demand_effective_rank_is_j(j):
    """D uniform over j experts has entropy ln j, so exp(H) = j and m = max(k, j). An
    integer effective rank sits 1e-9 (the snap distance) below the point where the size
    would become j + 1, so its decision margin is 1e-9, not 0 (for j < k the floor at k
    makes that point irrelevant)."""
    E, k = 16, 2
    l = np.full((5, E), -1000.0, dtype=np.float32)
    l[:, :j] = 0.0
    sel = O.select_tree(l, np.array([0, 1, 1, 2, 2]), k, [1.0, 0.6, 0.3], mode=O.ACCEPT,
                        pool_all=True)
    assert sel["m"] == max(k, j)
    assert sel["r"] == pytest.approx(j, rel=1e-14)
    if j >= k:
        assert sel["margin_rank"] == pytest.approx(1e-9, rel=1e-4)
    else:
        assert sel["margin_rank"] > 0.5


# ------------------------------------------- the size rule and the decision margins

SNAP = 1e-9  # the set-size reading: exp(H) within 1e-9 (relative) of an integer is it


def _size_rule(r, k, pool):
    """The reading of the pages' self-sizing taken here, as a rule on a number:
    m = n if |r - n| <= 1e-9 r for the nearest integer n, else ceil(r); floor k, cap pool."""
    n = round(r)
    m = n if abs(r - n) <= SNAP * r else math.ceil(r)
    return min(max(m, k), pool)


def _flip_distance(r, k, pool):
    """Brute force: the smallest relative change of r that changes _size_rule, found by a
    geometric scan then bisection on each side (inf when none below 1/r)."""
    m0 = _size_rule(r, k, pool)
    best = math.inf
    for sgn in (1.0, -1.0):
        lo, hi = 0.0, None
        eps = 1e-16
        while eps < 1.0 / r:
            if _size_rule(r * (1 + sgn * eps), k, pool) != m0:
                hi = eps
                break
            lo, eps = eps, eps * 1.25
        if hi is None:
            continue
        for _ in range(200):
            mid = 0.5 * (lo + hi)
            if _size_rule(r * (1 + sgn * mid), k, pool) != m0:
                hi = mid
            else:
                lo = mid
        best = min(best, hi)
    return best


def _two_level_demand(a, w):
    """One-hot routing that makes the demand exactly (1, ..., 1 [a times], w): nodes
    0..a-1 at depth 0 each routed to their own expert, node a at depth 1 (c = w) routed
    to expert a; k = 1."""
    E = a + 3
    hot = list(range(a + 1))
    depth = np.array([0] * a + [1], np.int32)
    return _one_hot_logits(hot, E), depth, [1.0, w]


@pytest.mark.parametrize("a,w,m_expect", [(5, 1e-13, 5), (5, 1e-6, 6), (12, 1e-12, 12),
                                          (12, 1e-5, 13), (3, 1.0, 4), (7, 0.25, 8)])
def test_effective_rank_closed_form_and_snap(a, w, m_expect):
    """D = (1 x a, w): q = (1/T x a, w/T) with T = a + w, so exp(H) = T * w^(-w/T), which
    lies just above a for small w. A distance to a below 1e-9 relative snaps to m = a
    (w = 1e-13: r - a ~ 3e-12); beyond it m = ceil(r) = a + 1 (w = 1e-6: r - a ~ 1.5e-5)."""
    l, depth, c = _two_level_demand(a, w)
    sel = O.select_tree(l, depth, 1, c, mode=O.ACCEPT, pool_all=True)
    T = a + w
    assert sel["r"] == pytest.approx(T * w ** (-w / T), rel=1e-13)
    assert sel["m"] == m_expect == _size_rule(sel["r"], 1, l.shape[1])


@pytest.mark.parametrize("a,w,k", [(5, 1e-13, 1), (5, 1e-6, 1), (12, 3e-11, 1), (3, 1.0, 1),
                                   (6, 0.4, 9), (6, 0.4, 2)])
def test_rank_margin_is_distance_to_the_size_flip(a, w, k):
    """margin_rank = the relative change of exp(H) that would change the set size, found
    here by bisection on the size rule itself (k = 9 floors every nearby size: +inf)."""
    l, depth, c = _two_level_demand(a, w)
    sel = O.select_tree(l, depth, k, c, mode=O.ACCEPT, pool_all=True)
    ref = _flip_distance(sel["r"], k, l.shape[1])
    if math.isinf(ref):
        assert sel["margin_rank"] > 1.0 / sel["r"] or math.isinf(sel["margin_rank"])
    else:
        assert sel["margin_rank"] == pytest.approx(ref, rel=1e-6, abs=1e-15)


def _fill_prune_brute(sel_noprune, l, k, anchor=True, pool_all=False, res=None, budget=0,
                      min_set=0):
    """Fill and prune cut gaps by sorting: the candidates (pool minus anchor) in
    (D desc, id asc) order, the first m - |anchor| taken; the removable members in
    (D asc, id asc) order, the first `removed` dropped."""
    D = sel_noprune["D"]
    nat, _ = O.topk(l, k)
    A = set(nat[0].tolist()) if anchor else set()
    pool = set(range(l.shape[1])) if pool_all else set(nat.ravel().tolist())
    cand = sorted(pool - A, key=lambda e: (-D[e], e))
    F = sel_noprune["m"] - len(A)
    fill = (D[cand[F - 1]] - D[cand[F]]) / D[cand[F - 1]] if 0 < F < len(cand) else math.inf
    prune = math.inf
    if res is not None:
        S = set(np.flatnonzero(sel_noprune["eligible"]).tolist())
        rem = sorted([e for e in S - A if not res[e]], key=lambda e: (D[e], e))
        r = min(budget, max(0, sel_noprune["m"] - max(min_set, k)), len(rem))
        if 0 < r < len(rem):
            prune = (D[rem[r]] - D[rem[r - 1]]) / D[rem[r]]
    return fill, prune


@pytest.mark.parametrize("seed", range(12))
def test_fill_and_prune_margins_by_sorting(seed):
    """margin_fill and margin_prune equal the relative demand gaps at the two cut points,
    recomputed by sorting the demand (catches a gap taken at the wrong rank or with the
    wrong sign)."""
    E, k = 32, 2
    t = W.eagle_tree(40 + seed)
    l = W.synthetic_logits(50 + seed, t.parent, E, 2.0 + 0.2 * seed)
    res = W.residency_mask(seed, E, 10)
    budget, min_set = 1 + seed % 4, 3 + seed % 5
    base = O.select_tree(l, t.depth, k, W.C_EAGLE, mode=O.ACCEPT)
    sel = O.select_tree(l, t.depth, k, W.C_EAGLE, mode=O.ACCEPT, prune=True, resident=res,
                        budget=budget, min_set=min_set)
    fill, prune = _fill_prune_brute(base, l, k, res=res, budget=budget, min_set=min_set)
    for got, ref in ((sel["margin_fill"], fill), (sel["margin_prune"], prune)):
        if math.isinf(ref):
            assert math.isinf(got)
        else:
            assert got == pytest.approx(ref, rel=1e-12)
    assert sel["margin_fill"] > 0 and sel["margin_prune"] > 0


def test_hand_built_fill_and_prune_cuts():
    """Demand (one-hot routing, c = 1 at every depth) = (4, 3, 2.5, 2, 1, 0.5) on experts
    0..5, k = 1, anchor = expert 0 (the root's), FIXED_B m = 4: the fill takes experts 1, 2,
    3 and leaves 4: gap (2 - 1) / 2 = 0.5. Pruning with experts 1, 3 non-resident, budget 1,
    min_set 2: removes expert 3 (the lowest removable), next is 1: gap (3 - 2) / 3."""
    E = 8
    counts = {0: 8, 1: 6, 2: 5, 3: 4, 4: 2, 5: 1}  # half-units: D = count / 2
    hot = [e for e, n in counts.items() for _ in range(n)]
    depth = np.zeros(len(hot), np.int32)
    l = _one_hot_logits(hot, E)
    c = [0.5]
    sel = O.select_tree(l, depth, 1, c, mode=O.FIXED_B, fixed_B=4)
    np.testing.assert_array_equal(sel["D"][:6], [4, 3, 2.5, 2, 1, 0.5])
    assert np.flatnonzero(sel["eligible"]).tolist() == [0, 1, 2, 3]
    assert sel["margin_fill"] == pytest.approx(0.5, rel=1e-15)
    assert math.isinf(sel["margin_prune"]) and math.isnan(sel["r"])
    res = np.array([1, 0, 1, 0, 1, 1, 1, 1], np.uint8)
    sel = O.select_tree(l, depth, 1, c, mode=O.FIXED_B, fixed_B=4, prune=True, resident=res,
                        budget=1, min_set=2)
    assert np.flatnonzero(sel["eligible"]).tolist() == [0, 1, 2] and sel["pruned"] == 1
    assert sel["margin_prune"] == pytest.approx(1.0 / 3.0, rel=1e-15)


def test_restricted_route_brute_force_and_identity():
    """The re-routing step on its own: with every expert allowed it is the natural top-k
    with softmax gates over the chosen logits; with a mask it is the unique best k-subset
    of the allowed experts (brute force), in descending order."""
    rng = np.random.Generator(np.random.PCG64(21))
    l = rng.standard_normal((7, 12)).astype(np.float32)
    idx, gates = O.restricted_route(l, np.ones(12), 3)
    nat, _ = O.topk(l, 3)
    np.testing.assert_array_equal(idx, nat)
    for r in range(7):
        np.testing.assert_allclose(gates[r], sp_softmax(l[r, idx[r]].astype(np.float64)),
                                   rtol=1e-13)
    allowed = np.zeros(12)
    allowed[[1, 4, 5, 8, 10]] = 1
    idx, _ = O.restricted_route(l, allowed, 3)
    for r in range(7):
        best = max(itertools.combinations([1, 4, 5, 8, 10], 3),
                   key=lambda T: sum(float(l[r, e]) for e in T))
        assert set(idx[r].tolist()) == set(best)
        assert all(l[r, idx[r][i]] >= l[r, idx[r][i + 1]] for i in range(2))
    with pytest.raises(ValueError):
        O.restricted_route(l, np.eye(12)[0], 3)


def test_root_only_commitment_gives_root_softmax():
    rng = np.random.Generator(np.random.PCG64(9))
    l = rng.standard_normal((9, 16)).astype(np.float32)
    sel = O.select_tree(l, W.tiny_tree().depth, 2, [1.0, 0.0], mode=O.ACCEPT)
    np.testing.assert_allclose(sel["D"], sp_softmax(l[0].astype(np.float64)), rtol=1e-14)


def test_all_equal_logits_selected_equals_natural():
    E, k = 16, 2
    l = np.zeros((9, E), dtype=np.float32)
    sel = O.select_tree(l, W.tiny_tree().depth, k, W.C_TINY, mode=O.ACCEPT)
    nat = O.select_tree(l, W.tiny_tree().depth, k, W.C_TINY, mode=O.NATURAL)
    # demand is uniform over all E, exp(H) = E, so m is capped at the pool (= U)
    assert sel["m"] == sel["union_nat"] == k
    np.testing.assert_array_equal(sel["idx"], nat["idx"])


def test_gates_are_softmax_of_chosen_logits():
    rng = np.random.Generator(np.random.PCG64(11))
    t = W.eagle_tree(3)
    l = W.synthetic_logits(4, t.parent, 32, 3.0)
    for mode in (O.NATURAL, O.ACCEPT):
        sel = O.select_tree(l, t.depth, 4, W.C_EAGLE, mode=mode)
        for n in range(t.N):
            ref = sp_softmax(l[n, sel["idx"][n]].astype(np.float64))
            np.testing.assert_allclose(sel["gates"][n], ref, rtol=1e-13)


# ----------------------------------------------------------------- brute force

def _tiny_case(seed, E=16, k=2, scale=3.0):
    t = W.tiny_tree()
    return W.synthetic_logits(seed, t.parent, E, scale), t.depth


@pytest.mark.parametrize("seed", range(20))
def test_anchor_fill_brute_force(seed):
    """S is the unique size-m superset of the root's natural top-k inside the pool
    that maximises the summed demand (distinct demands)."""
    k = 2
    l, depth = _tiny_case(seed)
    sel = O.select_tree(l, depth, k, W.C_TINY, mode=O.ACCEPT)
    nat, _ = O.topk(l, k)
    anchor = set(nat[0].tolist())
    pool = sorted(set(nat.ravel().tolist()))
    D = sel["D"]
    m = sel["m"]
    rest = [e for e in pool if e not in anchor]
    best, best_sum = None, -1.0
    for comb in itertools.combinations(rest, m - k):
        s = sum(D[e] for e in comb)
        if s > best_sum:
            best, best_sum = set(comb) | anchor, s
    assert set(np.flatnonzero(sel["eligible"]).tolist()) == best


@pytest.mark.parametrize("seed", range(20))
def test_prune_brute_force_and_invariants(seed):
    k, budget, min_set = 2, 3, 4
    t = W.eagle_tree(seed)
    l = W.synthetic_logits(seed, t.parent, 16, 1.5)
    res = W.residency_mask(seed, 16, 6)
    base = O.select_tree(l, t.depth, k, W.C_EAGLE, mode=O.ACCEPT)
    sel = O.select_tree(l, t.depth, k, W.C_EAGLE, mode=O.ACCEPT, prune=True, resident=res,
                        budget=budget, min_set=min_set)
    S0 = set(np.flatnonzero(base["eligible"]).tolist())
    S1 = set(np.flatnonzero(sel["eligible"]).tolist())
    anchor = set(O.topk(l[:1], k)[0][0].tolist())
    removed = S0 - S1
    assert S1 <= S0 and anchor <= S1
    assert len(removed) == sel["pruned"] <= budget
    assert all(res[e] == 0 for e in removed)
    assert len(S1) >= min(len(S0), max(min_set, k))
    removable = [e for e in S0 - anchor if res[e] == 0]
    r = min(budget, max(0, len(S0) - max(min_set, k)), len(removable))
    D = sel["D"]
    best = min(itertools.combinations(removable, r), key=lambda cmb: sum(D[e] for e in cmb))
    assert removed == set(best)


@pytest.mark.parametrize("seed", range(10))
def test_restricted_topk_brute_force(seed):
    k = 2
    l, depth = _tiny_case(seed, scale=2.0)
    sel = O.select_tree(l, depth, k, W.C_TINY, mode=O.ACCEPT)
    S = np.flatnonzero(sel["eligible"]).tolist()
    nat, _ = O.topk(l, k)
    for n in range(l.shape[0]):
        cands = [T for T in itertools.combinations(S, k)
                 if min(l[n, list(T)]) > max([l[n, e] for e in S if e not in T], default=-np.inf)]
        assert len(cands) == 1
        got = sel["idx"][n].tolist()
        assert set(got) == set(cands[0])
        assert all(l[n, got[i]] >= l[n, got[i + 1]] for i in range(k - 1))
        if set(nat[n].tolist()) <= set(S):
            assert got == nat[n].tolist()


def test_fixed_budget_mode_sets_size():
    t = W.eagle_tree(2)
    l = W.synthetic_logits(2, t.parent, 64, 3.0)
    for B in (4, 10, 30, 1000):
        sel = O.select_tree(l, t.depth, 4, W.C_EAGLE, mode=O.FIXED_B, fixed_B=B)
        assert sel["m"] == min(max(B, 4), sel["union_nat"])
        assert int(sel["eligible"].sum()) == sel["m"]


@pytest.mark.parametrize("scale", [1.0, 4.5])
def test_invariants_on_eagle_trees(scale):
    """Root's natural experts always eligible, |S| >= k, and the selected union
    never exceeds the natural union (it lies inside S, which lies inside U)."""
    E, k = 128, 8
    for seed in range(8):
        t = W.eagle_tree(100 + seed)
        l = W.synthetic_logits(seed, t.parent, E, scale)
        sel = O.select_tree(l, t.depth, k, W.C_EAGLE, mode=O.ACCEPT)
        nat, _ = O.topk(l, k)
        S = set(np.flatnonzero(sel["eligible"]).tolist())
        assert set(nat[0].tolist()) <= S
        assert len(S) >= k
        assert set(np.unique(sel["idx"]).tolist()) <= S <= set(np.unique(nat).tolist())
        assert sel["union_sel"] <= sel["union_nat"]


def test_permute_brute_force():
    for seed, (R, E, k, skew) in enumerate([(65, 128, 8, 0.0), (9, 16, 2, 1.0), (300, 32, 4, 1.2)]):
        idx = W.random_assignments(seed, R, E, k, skew)
        counts, offsets, perm = O.permute(idx, E)
        keys = sorted((int(idx[r, j]), r, j) for r in range(R) for j in range(k))
        assert perm.tolist() == [r * k + j for (_, r, j) in keys]
        np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))
        assert offsets[0] == 0 and offsets[-1] == R * k
        np.testing.assert_array_equal(np.diff(offsets), counts)


# ---------------------------------------------------------------- expert math

@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_single_expert_is_dense_swiglu(dt):
    """k = 1 reduces the layer to one dense SwiGLU FFN per token:
    y = W_down (silu(W_gate x) * (W_up x)), checked with torch fp64 + F.silu.
    f != d catches a transposed operand."""
    shape = W.LayerShape(d=48, E=3, k=1, f=20, dtype="fp32" if dt == torch.float32 else "bf16")
    wg, wu, wd = W.expert_weights(1, shape, std=0.2)
    g = torch.Generator().manual_seed(3)
    x = torch.randn(5, 48, generator=g).to(dt)
    idx = np.array([[0], [2], [1], [2], [0]], dtype=np.int32)
    got = O.moe_combine(x, wg, wu, wd, idx, np.ones((5, 1)))
    xd = x.double()
    for r in range(5):
        e = int(idx[r, 0])
        h = torch.nn.functional.silu(wg[e].double() @ xd[r]) * (wu[e].double() @ xd[r])
        np.testing.assert_allclose(got[r], (wd[e].double() @ h).numpy(), rtol=1e-11, atol=1e-13)


def test_gated_combine_weights_slots():
    shape = W.LayerShape(d=32, E=4, k=2, f=24, dtype="fp32")
    wg, wu, wd = W.expert_weights(2, shape, std=0.3)
    x = torch.randn(3, 32, generator=torch.Generator().manual_seed(1))
    idx = np.array([[1, 3], [0, 1], [2, 0]], dtype=np.int32)
    gates = np.array([[0.7, 0.3], [0.5, 0.5], [0.1, 0.9]])
    got = O.moe_combine(x, wg, wu, wd, idx, gates, rows=[2, 0])
    for q, r in enumerate([2, 0]):
        ref = np.zeros(32)
        for j in range(2):
            e = int(idx[r, j])
            h = torch.nn.functional.silu(wg[e].double() @ x[r].double()) * (wu[e].double() @ x[r].double())
            ref += gates[r, j] * (wd[e].double() @ h).numpy()
        np.testing.assert_allclose(got[q], ref, rtol=1e-11, atol=1e-13)


def test_forward_composes_router_selection_and_experts():
    shape = W.TINY
    t = W.tiny_tree()
    x = W.hidden_states(1, t.parent, shape.d, torch.float32)
    wr = W.router_weight(2, shape, std=0.1)
    wg, wu, wd = W.expert_weights(3, shape)
    out = O.forward(x, wr, wg, wu, wd, t.depth, shape.k, W.C_TINY, mode=O.ACCEPT)
    np.testing.assert_allclose(out["logits"], (x.double() @ wr.double().T).numpy(), rtol=1e-12)
    sel = O.select_tree(out["logits32"], t.depth, shape.k, W.C_TINY, mode=O.ACCEPT)
    np.testing.assert_array_equal(out["idx"], sel["idx"])
    y = O.moe_combine(x, wg, wu, wd, sel["idx"], sel["gates"])
    np.testing.assert_array_equal(out["y"], y)


# ------------------------------------------------- cost-aware draft selection

def _footprints(seed, cand, E, k, scale=2.0):
    logits = W.synthetic_logits(seed, cand.parent, E, scale)
    fp, _ = O.topk(logits, k)
    return fp


def test_draft_select_without_cost_is_top_by_probability():
    """lambda = 0 leaves only log P: cumulative log-probability falls along every edge,
    so the greedy tree is the root plus the gamma - 1 most probable candidates, taken in
    descending probability (the confidence-ordered tree)."""
    cand = W.eagle_candidates(5)
    fp = _footprints(5, cand, 64, 4)
    sel, _ = O.draft_select(cand.parent, cand.logp, fp, 64, 0.0, 65)
    order = sorted(range(1, cand.C), key=lambda v: (-float(cand.logp[v]), v))[:64]
    assert sel.tolist() == [0] + order


def test_draft_select_hand_example():
    """root {0,1}; a (log P -0.5, {2,3}) and b (-0.7, {0,1}) under the root; c (-0.55, {2,3})
    under a; d (-1.0, {1,5}) under b. gamma = 3.
    lambda = 0: a (-0.5), then c (-0.55)  -> S = {root, a, c}, union {0,1,2,3}.
    lambda = 0.2: b scores -0.7 > a's -0.5 - 0.4 = -0.9, so b; then a (-0.9) beats
    d (-1.0 - 0.2 = -1.2) and is taken                  -> S = {root, b, a}, union {0,1,2,3}.
    lambda = 0.6: b (-0.7); then a (-1.7) vs d (-1.6): d -> S = {root, b, d}, union {0,1,5}."""
    parent = np.array([-1, 0, 0, 1, 2], np.int32)          # root, a, b, c, d
    logp = np.array([0.0, -0.5, -0.7, -0.55, -1.0], np.float32)
    fp = np.array([[0, 1], [2, 3], [0, 1], [2, 3], [1, 5]], np.int32)
    s0, u0 = O.draft_select(parent, logp, fp, 8, 0.0, 3)
    s1, u1 = O.draft_select(parent, logp, fp, 8, 0.2, 3)
    s2, u2 = O.draft_select(parent, logp, fp, 8, 0.6, 3)
    assert (s0.tolist(), u0) == ([0, 1, 3], 4)
    assert (s1.tolist(), u1) == ([0, 2, 1], 4)
    assert (s2.tolist(), u2) == ([0, 2, 4], 3)


def test_draft_select_cost_is_a_set_difference():
    """The cost term counts experts, not footprint entries: with a footprint {2, 2} the
    node adds one expert, and an id outside [0, E) adds none. Root {0}; a (-0.5, {2, 2})
    and b (-0.45, {3, 4}) under the root; c (-0.6, {9, -1}) under the root, E = 8.
    lambda = 0.1: a scores -0.6, b -0.65, c -0.6 (no valid new expert): a (lower index
    than c on the tie) -> then c (-0.6) beats b (-0.65): S = {root, a, c}, union {0, 2}.
    Counting entries instead would give a -0.7 and pick c first."""
    parent = np.array([-1, 0, 0, 0], np.int32)
    logp = np.array([0.0, -0.5, -0.45, -0.6], np.float32)
    fp = np.array([[0, 0], [2, 2], [3, 4], [9, -1]], np.int32)
    sel, u = O.draft_select(parent, logp, fp, 8, 0.1, 3)
    assert (sel.tolist(), u) == ([0, 1, 3], 2)


@pytest.mark.parametrize("seed", range(6))
def test_draft_select_invariants(seed):
    """Ancestor-closed selection of gamma nodes, union = |union of the chosen footprints|,
    and with a huge lambda every step takes a candidate adding the fewest new experts."""
    E, k = 64, 4
    cand = W.eagle_candidates(100 + seed)
    fp = _footprints(seed, cand, E, k)
    for lam in (0.0, 0.3, 1e6):
        sel, u = O.draft_select(cand.parent, cand.logp, fp, E, lam, 65)
        assert len(sel) == 65 and len(set(sel.tolist())) == 65 and sel[0] == 0
        pos = {v: i for i, v in enumerate(sel.tolist())}
        assert all(pos[int(cand.parent[v])] < pos[v] for v in sel[1:].tolist())
        assert u == len(set(fp[sel].ravel().tolist()))
        if lam == 1e6:
            covered = set(fp[0].tolist())
            chosen = {0}
            for v in sel[1:].tolist():
                elig = [c for c in range(1, cand.C) if c not in chosen and
                        int(cand.parent[c]) in chosen]
                new = lambda c: len(set(fp[c].tolist()) - covered)  # noqa: E731
                assert new(v) == min(new(c) for c in elig)
                chosen.add(v)
                covered |= set(fp[v].tolist())
    # a cost weight never enlarges the covered set relative to the confidence order here
    s0, u0 = O.draft_select(cand.parent, cand.logp, fp, E, 0.0, 65)
    s1, u1 = O.draft_select(cand.parent, cand.logp, fp, E, 1e6, 65)
    assert u1 <= u0


# ---------------------------------------------------------------- pre-norm

def _bf16_value(bits: int) -> float:
    return float(torch.tensor([bits], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
                 .double()[0]) if bits < 0x8000 else -_bf16_value(bits & 0x7FFF)


def test_round_bf16_is_nearest_with_ties_to_even():
    """Brute force over the two neighbours: the result is never farther from v than the
    bf16 values one step either side, across normal and subnormal magnitudes; on the
    exact midpoint between two bf16 values the even significand wins."""
    rng = np.random.default_rng(0)
    mags = np.ldexp(rng.uniform(0.5, 1.0, 4000), rng.integers(-140, 128, 4000))
    vals = np.concatenate([mags, -mags[:1000]])
    for v in vals:
        b = O.round_bf16(v)
        got = _bf16_value(b)
        assert math.copysign(1.0, got) == math.copysign(1.0, v) or got == 0.0
        mag = b & 0x7FFF
        for nb in (mag - 1, mag + 1):
            if 0 <= nb < 0x7F80:
                alt = math.copysign(_bf16_value(nb), v)
                assert abs(v - got) <= abs(v - alt), (v, hex(b), hex(nb))
    # midpoints between consecutive bf16 values (exact in fp64)
    for mag in list(range(1, 200)) + list(range(0x3F00, 0x3F40)) + list(range(0x7F00, 0x7F7F)):
        lo, hi = _bf16_value(mag), _bf16_value(mag + 1)
        mid = (lo + hi) / 2
        want = mag if mag % 2 == 0 else mag + 1
        assert O.round_bf16(mid) == want
        assert O.round_bf16(-mid) == 0x8000 | want
        assert O.round_bf16(np.nextafter(mid, 0)) == mag
        assert O.round_bf16(np.nextafter(mid, np.inf)) == mag + 1


def test_round_bf16_matches_torch_on_fp32_inputs():
    """For values that are fp32 numbers a single rounding to bf16 is what torch's
    fp32 -> bf16 conversion (nearest, ties to even) does."""
    rng = np.random.default_rng(1)
    f = np.concatenate([rng.standard_normal(3000).astype(np.float32),
                        (rng.standard_normal(1000) * 1e-38).astype(np.float32),
                        np.float32([0.0, -0.0, 1.00390625, 1.01171875, 3.4e38])])
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([O.round_bf16(float(v)) for v in f], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)
    # past the largest finite bf16 by at least half a step: infinity
    assert O.round_bf16(2.0 ** 128) == 0x7F80
    assert O.round_bf16(-(2.0 ** 128)) == 0xFF80
    assert O.round_bf16(float(np.ldexp(511, 119))) == 0x7F80   # the midpoint rounds up to inf
    assert O.round_bf16(float(np.ldexp(509, 119))) == 0x7F7E   # midpoint, even side


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_rmsnorm_closed_form(dtype):
    """The unrounded pre-norm is x / sqrt(mean(x^2) + eps) (torch fp64); each row's mean
    square is then m / (m + eps); the stored values are that rounded once to the dtype;
    a row scaled by a power of two (eps negligible) normalises to the same output."""
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(7, 96, generator=g) * torch.tensor([1e-3, 0.02, 1, 30, 1, 1, 1])[:, None])
    x = x.to(dtype)
    x[5] = 0.0
    out, x64 = O.rmsnorm(x, unrounded=True)
    xd = x.double()
    ms = (xd ** 2).mean(1, keepdim=True)
    ref = xd / torch.sqrt(ms + O.NORM_EPS)
    np.testing.assert_allclose(x64, ref.numpy(), rtol=1e-14, atol=0)
    assert np.all(x64[5] == 0.0)
    got_ms = (x64 ** 2).mean(1)
    want_ms = (ms / (ms + O.NORM_EPS)).numpy()[:, 0]
    np.testing.assert_allclose(got_ms, want_ms, rtol=1e-12)
    if dtype == torch.bfloat16:
        assert out.dtype == np.uint16
        want = np.array([O.round_bf16(v) for v in x64.ravel()], dtype=np.uint16)
        np.testing.assert_array_equal(out.ravel(), want)
    else:
        np.testing.assert_array_equal(out, x64.astype(np.float32))
    x2 = x.clone()
    x2[3] = x[3] * 4.0
    out2 = O.rmsnorm(x2)
    np.testing.assert_array_equal(out2[3], out[3])
