"""Seeded random layer configurations through the whole layer, against the oracle.

Each case draws a layer (dtype, d, f, E, k), a block of B draft trees of one random
shape, a routing rule (natural, AcceptMoE, fixed size; with or without the root anchor;
with or without residency-aware pruning on a random residency mask), a router scale and
an expert path, then runs moe_tree_forward once and checks, as the whole-layer parity
tests do: router logits within 1e-4 of the row's largest |logit|; the selection tree by
tree against the fp64 oracle on the device's logits (a tree whose fp64 decision margin is
a tie is checked for validity instead); counts and offsets exactly; every row of y against
the oracle's experts and combine on the device's routing (2e-2 * max|ref| for bf16, 1e-4
for fp32). The cases cover expert counts that are not multiples of 32, k from 1 to 16,
blocks of one to three trees and trees of 2 to 65 nodes. A second set draws blocks of 4 to
80 trees of one random shape (up to ~5000 rows), with the router and y checked on sampled
rows. A third set draws tree sizes from 1 to 1000 nodes, blocks of up to 100 trees, layer
widths in steps of 64, and the pre-norm and residual options. In these three sets half the
cases hold the tensor-core expert kernel to 8-151 CTAs, where it pairs weight tiles over
row tiles of 32-128 tokens at any number of units. Two more sets draw offloaded
layers (against the resident layer, bit for bit) and draft selections (against the oracle),
and a last set routes junk expert ids through the experts.
"""
import numpy as np
import pytest
import torch

from expert_select_gb300 import moetree as M
from expert_select_gb300 import workload as W
from oracle import oracle as O
from test_gpu_parity import _check_selection, _sel_tree_from_oracle, _tree_of

pytestmark = pytest.mark.gpu
DEV = "cuda"
NF = M.MOE_INFO_FIELDS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from expert_select_gb300 import build
    build.build()
    M.lib()


def _cta_cap(rng):
    """The tensor-core expert kernel's CTA cap for a case: half the cases run on 8-151 CTAs,
    where the kernel takes weight-tile pairs at any number of units (on every SM the few
    units of a small layer stay single), the rest on one CTA per SM. Drawn last, so the
    other draws of a seed stay as they were."""
    return int(rng.integers(8, 152)) if rng.random() < 0.5 else 0


def _draw(seed):
    rng = np.random.default_rng(7000 + seed)
    dtype = "bf16" if rng.random() < 0.7 else "fp32"
    d = int(rng.choice([64, 128, 192, 256, 384]))
    f = int(rng.choice([64, 128, 192, 256]))
    E = int(rng.choice([8, 16, 24, 32, 48, 64, 100, 128, 160, 256]))
    k = int(rng.integers(1, min(16, E) + 1))
    B = int(rng.choice([1, 1, 2, 3]))
    steps = int(rng.integers(1, 6))
    topk = int(rng.integers(2, 11))
    most = topk + (steps - 1) * topk * topk
    tokens = int(min(rng.integers(1, 65), most))
    mode = str(rng.choice(["natural", "accept", "fixed"]))
    anchor = bool(rng.random() < 0.8)
    prune = mode != "natural" and bool(rng.random() < 0.4)
    std = float(rng.choice([0.02, 0.1, 0.3]))
    path = M.MOE_FFN_SIMT if (dtype == "fp32" or rng.random() < 0.25) else M.MOE_FFN_AUTO
    fixed_B = int(rng.integers(k, E + 1))
    min_set = int(rng.integers(k, max(k, 20) + 1))
    budget = int(rng.integers(0, 10))
    resident = (rng.random(E) < 0.5).astype(np.uint8)
    cap = _cta_cap(rng)
    return dict(dtype=dtype, d=d, f=f, E=E, k=k, B=B, steps=steps, topk=topk, tokens=tokens,
                mode=mode, anchor=anchor, prune=prune, std=std, path=path, fixed_B=fixed_B,
                min_set=min_set, budget=budget, resident=resident, cap=cap)


@pytest.mark.parametrize("seed", list(range(64)))
def test_random_layer_against_oracle(seed):
    c = _draw(seed)
    shape = W.LayerShape(d=c["d"], E=c["E"], k=c["k"], f=c["f"], dtype=c["dtype"])
    E, k, B = c["E"], c["k"], c["B"]
    trees = [W.eagle_tree(8000 + 17 * seed + b, steps=c["steps"], topk=c["topk"],
                          draft_tokens=c["tokens"]) for b in range(B)]
    N = trees[0].N
    assert all(t.N == N for t in trees)
    depth = np.stack([t.depth for t in trees]).astype(np.int32)
    R = B * N
    x = torch.cat([W.hidden_states(8100 + 17 * seed + b, t.parent, shape.d, shape.torch_dtype)
                   for b, t in enumerate(trees)])
    wr = W.router_weight(8200 + seed, shape, std=c["std"], device=DEV)
    wg, wu, wd = W.expert_weights(8300 + seed, shape, device=DEV)
    mode = {"natural": M.MOE_ROUTE_NATURAL, "accept": M.MOE_ROUTE_ACCEPT,
            "fixed": M.MOE_ROUTE_FIXED_B}[c["mode"]]
    P = M.select_params(mode, W.C_EAGLE, anchor=c["anchor"], prune=c["prune"],
                        reroute_budget=c["budget"], min_set=c["min_set"],
                        fixed_B=c["fixed_B"] if c["mode"] == "fixed" else 0)
    L = M.layer_desc(shape.d, E, k, shape.f, shape.dtype)
    out = dict(logits=torch.empty(R, E, device=DEV),
               topk_idx=torch.empty(R, k, dtype=torch.int32, device=DEV),
               gates=torch.empty(R, k, device=DEV),
               eligible=torch.empty(B, E, dtype=torch.uint8, device=DEV),
               info=torch.empty(B, NF, dtype=torch.int32, device=DEV),
               counts=torch.empty(E, dtype=torch.int32, device=DEV),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV))
    res = torch.from_numpy(c["resident"]).to(DEV) if c["prune"] else None
    y = torch.full((R, shape.d), float("nan"), dtype=shape.torch_dtype, device=DEV)
    ws = M.workspace(L, B, N)
    M.moe_tree_forward(L, P, x.to(DEV), wr, wg, wu, wd, None,
                       torch.from_numpy(depth.reshape(-1).copy()).to(DEV), B, N, res, y, ws,
                       M.tree_outputs(**out), M.run_opts(c["path"], ffn_max_ctas=c["cap"]))
    torch.cuda.synchronize()
    assert M.moe_workspace_check(ws) == 0
    got = {key: v.cpu().numpy() for key, v in out.items()}
    # 1. the router against the oracle's own fp64 logits
    ref_l = O.router(x, wr.cpu())
    assert (np.abs(got["logits"] - ref_l) <= 1e-4 * np.abs(ref_l).max(axis=1, keepdims=True)).all()
    # 2. the selection, tree by tree, from the device's logits
    omode = {"natural": O.NATURAL, "accept": O.ACCEPT, "fixed": O.FIXED_B}[c["mode"]]
    kw = dict(mode=omode, c=W.C_EAGLE, anchor=c["anchor"])
    if c["mode"] == "fixed":
        kw["fixed_B"] = c["fixed_B"]
    if c["prune"]:
        kw.update(prune=True, resident=c["resident"], budget=c["budget"], min_set=c["min_set"])
    _check_selection(shape, kw, got["logits"], depth, got["topk_idx"], got["gates"],
                     got["eligible"], got["info"], N, B)
    # 3. the counting sort of the device's routing
    rc, ro, _ = O.permute(got["topk_idx"], E)
    np.testing.assert_array_equal(got["counts"], rc)
    np.testing.assert_array_equal(got["offsets"], ro)
    # 4. every row of y: the oracle's experts and combine on the device's routing
    ref_y = O.moe_combine(x, wg.cpu(), wu.cpu(), wd.cpu(), got["topk_idx"], got["gates"])
    tol = 2e-2 if shape.dtype == "bf16" else 1e-4
    err = np.abs(y.double().cpu().numpy() - ref_y).max()
    assert err <= tol * np.abs(ref_y).max(), (c, err)


def _draw_large(seed):
    rng = np.random.default_rng(9000 + seed)
    dtype = "bf16" if rng.random() < 0.85 else "fp32"
    d = int(rng.choice([256, 512, 1024]))
    f = int(rng.choice([128, 256, 384]))
    E = int(rng.choice([32, 64, 100, 128, 160, 256]))
    k = int(rng.integers(1, min(16, E) + 1))
    B = int(rng.integers(4, 81))
    steps = int(rng.integers(2, 6))
    topk = int(rng.integers(4, 11))
    tokens = int(min(rng.integers(16, 65), topk + (steps - 1) * topk * topk))
    mode = str(rng.choice(["natural", "accept", "accept", "fixed"]))
    prune = mode != "natural" and bool(rng.random() < 0.4)
    return dict(dtype=dtype, d=d, f=f, E=E, k=k, B=B, steps=steps, topk=topk, tokens=tokens,
                mode=mode, anchor=bool(rng.random() < 0.8), prune=prune,
                std=float(rng.choice([0.02, 0.1, 0.3])),
                fixed_B=int(rng.integers(k, E + 1)), min_set=int(rng.integers(k, max(k, 24) + 1)),
                budget=int(rng.integers(0, 10)), resident=(rng.random(E) < 0.5).astype(np.uint8),
                cap=_cta_cap(rng))


@pytest.mark.parametrize("seed", list(range(48)))
def test_random_large_block_against_oracle(seed):
    """Blocks of 4 to 80 trees (up to ~5000 rows) of random layers: the tensor-core router,
    the selection of many trees per launch (clusters, or one CTA per tree past three waves
    of clusters), the many-CTA permute, experts with hundreds of tokens in several row
    tiles; the same checks as above, y on 48 sampled rows."""
    c = _draw_large(seed)
    shape = W.LayerShape(d=c["d"], E=c["E"], k=c["k"], f=c["f"], dtype=c["dtype"])
    E, B = c["E"], c["B"]
    tree = W.eagle_tree(9100 + seed, steps=c["steps"], topk=c["topk"], draft_tokens=c["tokens"])
    N = tree.N
    depth = np.tile(tree.depth.astype(np.int32), (B, 1))
    R = B * N
    x = torch.cat([W.hidden_states(9200 + 131 * seed + b, tree.parent, shape.d,
                                   shape.torch_dtype) for b in range(B)])
    wr = W.router_weight(9300 + seed, shape, std=c["std"], device=DEV)
    wg, wu, wd = W.expert_weights(9400 + seed, shape, device=DEV)
    mode = {"natural": M.MOE_ROUTE_NATURAL, "accept": M.MOE_ROUTE_ACCEPT,
            "fixed": M.MOE_ROUTE_FIXED_B}[c["mode"]]
    P = M.select_params(mode, W.C_EAGLE, anchor=c["anchor"], prune=c["prune"],
                        reroute_budget=c["budget"], min_set=c["min_set"],
                        fixed_B=c["fixed_B"] if c["mode"] == "fixed" else 0)
    L = M.layer_desc(shape.d, E, shape.k, shape.f, shape.dtype)
    out = dict(logits=torch.empty(R, E, device=DEV),
               topk_idx=torch.empty(R, shape.k, dtype=torch.int32, device=DEV),
               gates=torch.empty(R, shape.k, device=DEV),
               eligible=torch.empty(B, E, dtype=torch.uint8, device=DEV),
               info=torch.empty(B, NF, dtype=torch.int32, device=DEV),
               counts=torch.empty(E, dtype=torch.int32, device=DEV),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV))
    res = torch.from_numpy(c["resident"]).to(DEV) if c["prune"] else None
    y = torch.full((R, shape.d), float("nan"), dtype=shape.torch_dtype, device=DEV)
    ws = M.workspace(L, B, N)
    M.moe_tree_forward(L, P, x.to(DEV), wr, wg, wu, wd, None,
                       torch.from_numpy(depth.reshape(-1).copy()).to(DEV), B, N, res, y, ws,
                       M.tree_outputs(**out), M.run_opts(M.MOE_FFN_AUTO, ffn_max_ctas=c["cap"]))
    torch.cuda.synchronize()
    assert M.moe_workspace_check(ws) == 0
    got = {key: v.cpu().numpy() for key, v in out.items()}
    rows = np.random.default_rng(seed).choice(R, min(R, 256), replace=False)
    ref_l = O.router(x[rows], wr.cpu())
    assert (np.abs(got["logits"][rows] - ref_l) <=
            1e-4 * np.abs(ref_l).max(axis=1, keepdims=True)).all()
    omode = {"natural": O.NATURAL, "accept": O.ACCEPT, "fixed": O.FIXED_B}[c["mode"]]
    kw = dict(mode=omode, c=W.C_EAGLE, anchor=c["anchor"])
    if c["mode"] == "fixed":
        kw["fixed_B"] = c["fixed_B"]
    if c["prune"]:
        kw.update(prune=True, resident=c["resident"], budget=c["budget"], min_set=c["min_set"])
    _check_selection(shape, kw, got["logits"], depth, got["topk_idx"], got["gates"],
                     got["eligible"], got["info"], N, B)
    rc, ro, _ = O.permute(got["topk_idx"], E)
    np.testing.assert_array_equal(got["counts"], rc)
    np.testing.assert_array_equal(got["offsets"], ro)
    sample = np.random.default_rng(seed + 1).choice(R, 48, replace=False).tolist()
    ref_y = O.moe_combine(x, wg.cpu(), wu.cpu(), wd.cpu(), got["topk_idx"], got["gates"],
                          rows=sample)
    tol = 2e-2 if shape.dtype == "bf16" else 1e-4
    err = np.abs(y.double().cpu().numpy()[sample] - ref_y).max()
    assert err <= tol * np.abs(ref_y).max(), (c, err)


def _draw_wide(seed):
    rng = np.random.default_rng(50000 + seed)
    dtype = "bf16" if rng.random() < 0.8 else "fp32"
    d = int(64 * rng.integers(1, 33))
    f = int(64 * rng.integers(1, 17))
    E = int(rng.integers(8, 257))
    k = int(rng.integers(1, min(16, E) + 1))
    big = rng.random() < 0.3
    N = int(rng.integers(257, 1001)) if big else int(rng.integers(1, 257))
    B = 1 if big else int(rng.integers(1, 101 if N <= 65 else 9))
    mode = str(rng.choice(["natural", "accept", "accept", "fixed"]))
    prune = mode != "natural" and bool(rng.random() < 0.4)
    return dict(dtype=dtype, d=d, f=f, E=E, k=k, N=N, B=B, mode=mode,
                anchor=bool(rng.random() < 0.8), prune=prune,
                std=float(rng.choice([0.02, 0.1, 0.3, 1.0])),
                fixed_B=int(rng.integers(k, E + 1)), min_set=int(rng.integers(k, max(k, 24) + 1)),
                budget=int(rng.integers(0, 10)), resident=(rng.random(E) < 0.5).astype(np.uint8),
                norm=bool(rng.random() < 0.3), residual=bool(rng.random() < 0.3),
                path=M.MOE_FFN_SIMT if (dtype == "fp32" or rng.random() < 0.15) else M.MOE_FFN_AUTO,
                cap=_cta_cap(rng))


@pytest.mark.parametrize("seed", list(range(48)))
def test_random_tree_sizes_and_options(seed):
    """Trees of 1 to 1000 nodes (past 256 the one-CTA selector), blocks of up to 100 trees,
    d up to 2048 and f up to 1024 in steps of 64, E from 8 to 256, both expert paths, the
    pre-norm and residual options; the selection of every tree, counts and offsets
    exactly, logits and y on sampled rows (y = x + MoE(rmsnorm(x)) with both options)."""
    c = _draw_wide(seed)
    shape = W.LayerShape(d=c["d"], E=c["E"], k=c["k"], f=c["f"], dtype=c["dtype"])
    E, B, N = c["E"], c["B"], c["N"]
    parent, depth1 = _tree_of(N, 60000 + seed)
    depth = np.tile(depth1.astype(np.int32), (B, 1))
    R = B * N
    x = torch.cat([W.hidden_states(61000 + 97 * seed + b, parent, shape.d, shape.torch_dtype)
                   for b in range(B)])
    wr = W.router_weight(62000 + seed, shape, std=c["std"], device=DEV)
    wg, wu, wd = W.expert_weights(63000 + seed, shape, device=DEV)
    mode = {"natural": M.MOE_ROUTE_NATURAL, "accept": M.MOE_ROUTE_ACCEPT,
            "fixed": M.MOE_ROUTE_FIXED_B}[c["mode"]]
    P = M.select_params(mode, W.C_EAGLE, anchor=c["anchor"], prune=c["prune"],
                        reroute_budget=c["budget"], min_set=c["min_set"],
                        fixed_B=c["fixed_B"] if c["mode"] == "fixed" else 0)
    L = M.layer_desc(shape.d, E, shape.k, shape.f, shape.dtype)
    out = dict(logits=torch.empty(R, E, device=DEV),
               topk_idx=torch.empty(R, shape.k, dtype=torch.int32, device=DEV),
               gates=torch.empty(R, shape.k, device=DEV),
               eligible=torch.empty(B, E, dtype=torch.uint8, device=DEV),
               info=torch.empty(B, NF, dtype=torch.int32, device=DEV),
               counts=torch.empty(E, dtype=torch.int32, device=DEV),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV))
    res = torch.from_numpy(c["resident"]).to(DEV) if c["prune"] else None
    y = torch.full((R, shape.d), float("nan"), dtype=shape.torch_dtype, device=DEV)
    ws = M.workspace(L, B, N)
    xd = x.to(DEV)
    M.moe_tree_forward(L, P, xd, wr, wg, wu, wd, None,
                       torch.from_numpy(depth.reshape(-1).copy()).to(DEV), B, N, res, y, ws,
                       M.tree_outputs(**out),
                       M.run_opts(c["path"], residual=c["residual"], norm_input=c["norm"],
                                  ffn_max_ctas=c["cap"]))
    torch.cuda.synchronize()
    assert M.moe_workspace_check(ws) == 0
    got = {key: v.cpu().numpy() for key, v in out.items()}
    if c["norm"]:
        xn = torch.empty_like(xd)
        M.moe_rms_norm(L, xd, xn)
        torch.cuda.synchronize()
        xr = xn.cpu()
    else:
        xr = x
    rows = np.random.default_rng(seed).choice(R, min(R, 128), replace=False)
    ref_l = O.router(xr[rows], wr.cpu())
    assert (np.abs(got["logits"][rows] - ref_l) <=
            1e-4 * np.abs(ref_l).max(axis=1, keepdims=True)).all()
    omode = {"natural": O.NATURAL, "accept": O.ACCEPT, "fixed": O.FIXED_B}[c["mode"]]
    kw = dict(mode=omode, c=W.C_EAGLE, anchor=c["anchor"])
    if c["mode"] == "fixed":
        kw["fixed_B"] = c["fixed_B"]
    if c["prune"]:
        kw.update(prune=True, resident=c["resident"], budget=c["budget"], min_set=c["min_set"])
    _check_selection(shape, kw, got["logits"], depth, got["topk_idx"], got["gates"],
                     got["eligible"], got["info"], N, B)
    rc, ro, _ = O.permute(got["topk_idx"], E)
    np.testing.assert_array_equal(got["counts"], rc)
    np.testing.assert_array_equal(got["offsets"], ro)
    sample = np.random.default_rng(seed + 1).choice(R, min(R, 24), replace=False).tolist()
    ref_y = O.moe_combine(xr, wg.cpu(), wu.cpu(), wd.cpu(), got["topk_idx"], got["gates"],
                          rows=sample)
    if c["residual"]:
        ref_y = ref_y + x.double().numpy()[sample]
    tol = 2e-2 if shape.dtype == "bf16" else 1e-4
    err = np.abs(y.double().cpu().numpy()[sample] - ref_y).max()
    assert err <= tol * np.abs(ref_y).max(), (c, err)


@pytest.mark.parametrize("seed", list(range(24)))
def test_random_offloaded_layer_equals_resident(seed):
    """The offloaded layer on random shapes, slot counts (k to E), routing rules, pruning,
    pre-norm and residual, blocks of 1-3 trees over three steps: output and routing equal
    to the resident layer's bit for bit, counters consistent."""
    rng = np.random.default_rng(70000 + seed)
    dtype = "bf16" if rng.random() < 0.7 else "fp32"
    d = int(64 * rng.integers(1, 9)); f = int(64 * rng.integers(1, 5))
    E = int(rng.integers(8, 97)); k = int(rng.integers(1, min(8, E) + 1))
    slots = int(rng.integers(k, E + 1))
    shape = W.LayerShape(d=d, E=E, k=k, f=f, dtype=dtype)
    mode = str(rng.choice(["natural", "accept", "fixed"]))
    prune = mode != "natural" and bool(rng.random() < 0.5)
    norm = bool(rng.random() < 0.4)
    std = float(rng.choice([0.02, 0.1, 0.3]))
    if mode == "natural":
        P = M.select_params(M.MOE_ROUTE_NATURAL, W.C_EAGLE)
    elif mode == "accept":
        P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE, prune=prune,
                            reroute_budget=int(rng.integers(0, 9)), min_set=int(rng.integers(k, k + 12)))
    else:
        P = M.select_params(M.MOE_ROUTE_FIXED_B, W.C_EAGLE, prune=prune,
                            reroute_budget=int(rng.integers(0, 9)), min_set=int(rng.integers(k, k + 12)),
                            fixed_B=int(rng.integers(k, E + 1)))
    wg, wu, wd = W.expert_weights(71000 + seed, shape, device=DEV)
    hg, hu, hd = (w.cpu().pin_memory() for w in (wg, wu, wd))
    pg = torch.zeros(slots, f, d, dtype=shape.torch_dtype, device=DEV)
    pu = torch.zeros_like(pg)
    pd = torch.zeros(slots, d, f, dtype=shape.torch_dtype, device=DEV)
    wr = W.router_weight(72000 + seed, shape, std=std, device=DEV)
    L = M.layer_desc(d, E, k, f, dtype)
    Ls = M.layer_desc(d, E, k, f, dtype, slots=slots)
    table = M.Residency(n_layers=1, E=E, slots=slots)
    side = torch.cuda.Stream()
    B = int(rng.integers(1, 4))
    for step in range(3):
        t = W.eagle_tree(73000 + 7 * seed + step, steps=int(rng.integers(1, 6)), topk=int(rng.integers(2, 11)),
                         draft_tokens=int(rng.integers(1, 65)))
        N = t.N
        x = torch.cat([W.hidden_states(74000 + 11 * seed + 3 * step + b, t.parent, d, shape.torch_dtype)
                       for b in range(B)]).to(DEV)
        dep = torch.from_numpy(np.tile(t.depth, B).astype(np.int32)).to(DEV)
        _, res_before = table.query(0)
        res_dev = torch.from_numpy(res_before.copy()).to(DEV)
        idx_ref = torch.empty(B * N, k, dtype=torch.int32, device=DEV)
        cnt_ref = torch.empty(E, dtype=torch.int32, device=DEV)
        y_ref = torch.empty(B * N, d, dtype=shape.torch_dtype, device=DEV)
        ws = M.workspace(L, B, N)
        opts = M.run_opts(norm_input=norm, residual=norm)
        M.moe_tree_forward(L, P, x, wr, wg, wu, wd, None, dep, B, N, res_dev, y_ref, ws,
                           M.tree_outputs(topk_idx=idx_ref, counts=cnt_ref), opts)
        idx = torch.empty_like(idx_ref)
        y = torch.full_like(y_ref, float("nan"))
        ws2 = M.workspace(Ls, B, N)
        st = M.moe_offload_forward(Ls, P, x, wr, hg, hu, hd, pg, pu, pd, table, 0, dep, B, N,
                                   y, ws2, M.tree_outputs(topk_idx=idx), opts=opts, side_stream=side)
        torch.cuda.synchronize()
        assert M.moe_workspace_check(ws2) == 0
        assert torch.equal(idx, idx_ref)
        assert torch.equal(y, y_ref), (seed, step)
        union = int((cnt_ref > 0).sum())
        assert st.needed == union and st.hits + st.uploads == union


@pytest.mark.parametrize("seed", list(range(48)))
def test_random_draft_selection_against_oracle(seed):
    """EcoSpec-style draft selection on random candidate pools (up to ~3200 candidates),
    E 4-256, k 1-16, lambda 0-5, gamma 1-300, with repeated and out-of-range footprint ids
    in a fifth of the cases: selection, parents, depths and union bit-exact."""
    rng = np.random.default_rng(80000 + seed)
    steps = int(rng.integers(1, 10)); topk = int(rng.integers(1, 21))
    cand = W.eagle_candidates(81000 + seed, steps=steps, topk=topk)
    C = cand.C
    E = int(rng.integers(4, 257)); k = int(rng.integers(1, min(16, E) + 1))
    junk = rng.random() < 0.2
    if junk:
        fp = rng.integers(-3, E + 3, size=(C, k)).astype(np.int32)
    else:
        fp = np.stack([rng.choice(E, size=k, replace=False) for _ in range(C)]).astype(np.int32)
    lam = float(rng.choice([0.0, 0.01, 0.1, 0.3, 1.0, 5.0]))
    gamma = int(rng.integers(1, min(C, 300) + 1))
    L = M.layer_desc(256, E, k, 128, "bf16")
    sel = torch.empty(gamma, dtype=torch.int32, device=DEV)
    spar, sdep = torch.empty_like(sel), torch.empty_like(sel)
    nu = torch.empty(1, dtype=torch.int32, device=DEV)
    td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    M.moe_draft_select(L, td(cand.parent), td(cand.depth), td(cand.logp), td(fp), lam, gamma,
                       sel, spar, sdep, n_union=nu)
    torch.cuda.synchronize()
    ref_sel, ref_u = O.draft_select(cand.parent, cand.logp, fp, E, lam, gamma)
    np.testing.assert_array_equal(sel.cpu().numpy(), ref_sel)
    rp, rd = _sel_tree_from_oracle(cand, ref_sel)
    np.testing.assert_array_equal(spar.cpu().numpy(), rp)
    np.testing.assert_array_equal(sdep.cpu().numpy(), rd)
    assert int(nu.item()) == ref_u


@pytest.mark.parametrize("seed", list(range(24)))
def test_random_junk_routing_through_the_experts(seed):
    """moe_expert_forward on routing with out-of-range ids (5% of slots) and repeated ids
    (5% of rows), 1 to 3000 rows, both expert paths: the check bit is set exactly when a
    slot is skipped, and y equals the oracle over the valid slots (the first slot of a
    repeated id)."""
    rng = np.random.default_rng(90000 + seed)
    dtype = "bf16" if rng.random() < 0.7 else "fp32"
    d = int(64 * rng.integers(1, 9)); f = int(64 * rng.integers(1, 5))
    E = int(rng.integers(4, 257)); k = int(rng.integers(1, min(16, E) + 1))
    R = int(rng.choice([1, 7, 65, 300, 1100, 3000]))
    shape = W.LayerShape(d=d, E=E, k=k, f=f, dtype=dtype)
    L = M.layer_desc(d, E, k, f, dtype)
    idx = W.random_assignments(91000 + seed, R, E, k, float(rng.choice([0.0, 1.0])))
    junk = rng.random(idx.shape) < 0.05
    idx[junk] = rng.integers(-5, E + 5, size=int(junk.sum()))
    if k > 1:  # some rows repeat their first id in a later slot
        rep = rng.random(R) < 0.05
        idx[rep, k - 1] = idx[rep, 0]
    gates = W.random_gates(92000 + seed, R, k)
    wg, wu, wd = W.expert_weights(93000 + seed, shape, device=DEV)
    x = W.hidden_states(94000 + seed, np.arange(-1, R - 1, dtype=np.int32), d, shape.torch_dtype)
    y = torch.full((R, d), float("nan"), dtype=shape.torch_dtype, device=DEV)
    ws = M.workspace(L, 1, R)
    path = M.MOE_FFN_SIMT if (dtype == "fp32" or rng.random() < 0.3) else M.MOE_FFN_TCGEN05
    M.moe_expert_forward(L, x.to(DEV), wg, wu, wd, None, torch.from_numpy(idx).to(DEV),
                         torch.from_numpy(gates).to(DEV), y, ws, M.run_opts(path))
    torch.cuda.synchronize()
    # the valid slots: in range, and the first slot of a repeated id
    valid = (idx >= 0) & (idx < E)
    for j in range(1, k):
        for q in range(j):
            valid[:, j] &= idx[:, j] != idx[:, q]
    bad = not valid.all()
    chk = M.moe_workspace_check(ws)
    assert chk == (1 if bad else 0), (chk, bad)
    g = np.where(valid, gates, 0.0).astype(np.float64)
    ii = np.where(valid, idx, 0).astype(np.int32)
    rows = np.random.default_rng(seed).choice(R, min(R, 24), replace=False).tolist()
    ref = O.moe_combine(x, wg.cpu(), wu.cpu(), wd.cpu(), ii, g, rows=rows)
    tol = 2e-2 if dtype == "bf16" else 1e-4
    err = np.abs(y.double().cpu().numpy()[rows] - ref).max()
    assert err <= tol * max(np.abs(ref).max(), 1e-30), (seed, err)
