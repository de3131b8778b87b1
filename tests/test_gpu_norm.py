"""GPU tests of the RMS pre-norm (moe_rms_norm, moe_run_opts.norm_input).

The pre-norm is a plain definition, x / sqrt(mean(x^2) + eps) per row, computed in fp64
on both sides and rounded once to the layer dtype, so the device's output must equal the
oracle's bit for bit. The two fp64 sums of squares run in different orders, so a value
within about 2^-45 (relative) of a rounding midpoint could round the other way; such an
element is excused if the device chose the other neighbour of that midpoint (none is
expected at these sizes).

The layer with norm_input routes and computes the experts on the normalised rows and
adds the original rows as the residual; the checks follow the whole-layer parity tests:
logits within 1e-4 of the row's largest |logit| of the oracle's, routing bit-exact from
the device's logits, sampled rows of y within 2e-2 * max|ref| (bf16).
"""
import numpy as np
import pytest
import torch

from expert_select_gb300 import moetree as M
from expert_select_gb300 import workload as W
from oracle import oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from expert_select_gb300 import build
    build.build()
    M.lib()


def _bits(t: torch.Tensor) -> np.ndarray:
    t = t.cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy().view(np.uint32)


def _values(bits: np.ndarray) -> np.ndarray:
    if bits.dtype == np.uint16:
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return bits.view(np.float32).astype(np.float64)


def _assert_norm_equal(got: torch.Tensor, x: torch.Tensor):
    want, x64 = O.rmsnorm(x, unrounded=True)
    gb = _bits(got)
    wb = want.view(np.uint16) if want.dtype == np.uint16 else want.view(np.uint32)
    bad = np.argwhere(gb != wb)
    for i in map(tuple, bad):
        a, b = _values(np.array([wb[i]]))[0], _values(np.array([gb[i]]))[0]
        mid = (a + b) / 2
        # neighbours on either side of a midpoint the exact value sits on
        assert abs(x64[i] - mid) <= 2.0 ** -44 * abs(x64[i]), (i, a, b, x64[i])
    assert len(bad) <= 2


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("R,d", [(1, 8), (37, 264), (300, 2048), (65, 2880), (4160, 2048)])
def test_rms_norm_matches_oracle(dtype, R, d):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(R * 7 + d)
    scale = torch.exp(torch.randn(R, 1, generator=g) * 3)  # row RMS from ~1e-4 to ~1e4
    x = (torch.randn(R, d, generator=g) * scale).to(tdt)
    L = M.layer_desc(d, 16, 2, 64, dtype)
    xd = x.to(DEV)
    xn = torch.full_like(xd, float("nan"))
    M.moe_rms_norm(L, xd, xn)
    torch.cuda.synchronize()
    _assert_norm_equal(xn, x)


def test_rms_norm_edge_rows():
    """Zero rows give zeros (eps keeps the scale finite); rows of huge and tiny bf16
    values normalise without overflow or underflow (the squares are summed in fp64);
    R = 0 launches nothing."""
    d = 2048
    L = M.layer_desc(d, 16, 2, 64, "bf16")
    x = torch.randn(6, d).to(torch.bfloat16)
    x[0] = 0
    x[1] *= 1e30
    x[2] *= 1e-30
    x[3, :] = 0
    x[3, 5] = 3.0  # a single nonzero element: sqrt(d) * sign
    x[4] = torch.finfo(torch.bfloat16).max
    x[5] = -torch.finfo(torch.bfloat16).tiny
    xd = x.to(DEV)
    xn = torch.empty_like(xd)
    M.moe_rms_norm(L, xd, xn)
    torch.cuda.synchronize()
    _assert_norm_equal(xn, x)
    got = xn.double().cpu()
    assert torch.all(got[0] == 0)
    assert torch.isfinite(got).all()
    assert abs(got[3, 5].item() - d ** 0.5) <= 2 ** -7 * d ** 0.5
    empty = torch.empty(0, d, dtype=torch.bfloat16, device=DEV)
    M.moe_rms_norm(L, empty, torch.empty_like(empty))


def _layer(shape, seed, std):
    wr = W.router_weight(seed, shape, std=std, device=DEV)
    wg, wu, wd = W.expert_weights(seed + 1, shape, device=DEV)
    return wr, wg, wu, wd


def test_norm_option_equals_the_explicit_norm():
    """moe_tree_forward with norm_input computes the same as moe_rms_norm followed by the
    layer on the normalised rows: equal routing and equal y bit for bit without the
    residual; with the residual, y = x + that output (one rounding apart)."""
    shape = W.QWEN3_30B_A3B
    B = 2
    parent, depth = W.tree_block(41, B, "eagle")
    N = parent.shape[1]
    R = B * N
    x = (W.hidden_states(42, parent, shape.d, torch.bfloat16).float() * 7.0).to(torch.bfloat16)
    x = x.to(DEV)
    wr, wg, wu, wd = _layer(shape, 43, 0.1)
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    dp = torch.from_numpy(depth.reshape(-1).copy()).to(DEV)
    ws = M.workspace(L, B, N)

    def run(inp, **kw):
        idx = torch.empty(R, shape.k, dtype=torch.int32, device=DEV)
        y = torch.empty(R, shape.d, dtype=torch.bfloat16, device=DEV)
        M.moe_tree_forward(L, P, inp, wr, wg, wu, wd, None, dp, B, N, None, y, ws,
                           M.tree_outputs(topk_idx=idx), M.run_opts(**kw))
        torch.cuda.synchronize()
        assert M.moe_workspace_check(ws) == 0
        return idx, y

    xn = torch.empty_like(x)
    M.moe_rms_norm(L, x, xn)
    i_ref, y_ref = run(xn)
    i_opt, y_opt = run(x, norm_input=True)
    assert torch.equal(i_opt, i_ref)
    assert torch.equal(y_opt, y_ref)
    i_res, y_res = run(x, norm_input=True, residual=True)
    assert torch.equal(i_res, i_ref)
    ref = x.double() + y_ref.double()
    assert (y_res.double() - ref).abs().max().item() <= 2 ** -7 * ref.abs().max().item()
    # the experts-only entry point takes the option too
    counts = torch.empty(shape.E, dtype=torch.int32, device=DEV)
    g = torch.empty(R, shape.k, device=DEV)
    idx2 = torch.empty_like(i_ref)
    M.moe_tree_forward(L, P, x, wr, wg, wu, wd, None, dp, B, N, None, y_opt, ws,
                       M.tree_outputs(topk_idx=idx2, gates=g, counts=counts),
                       M.run_opts(norm_input=True))
    y_ex = torch.empty_like(y_opt)
    M.moe_expert_forward(L, x, wg, wu, wd, None, idx2, g, y_ex, ws,
                         M.run_opts(norm_input=True))
    torch.cuda.synchronize()
    assert torch.equal(y_ex, y_opt)


@pytest.mark.parametrize("shape,std", [(W.QWEN3_30B_A3B, 0.02), (W.QWEN3_30B_A3B, 0.1),
                                       (W.LayerShape(d=2880, E=32, k=4, f=2880, dtype="bf16"),
                                        0.1)])
def test_normed_layer_against_oracle(shape, std):
    B = 2
    parent, depth = W.tree_block(51, B, "eagle")
    N = parent.shape[1]
    R = B * N
    x = (W.hidden_states(52, parent, shape.d, torch.bfloat16).float() * 5.0).to(torch.bfloat16)
    wr, wg, wu, wd = _layer(shape, 53, std)
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    dp = torch.from_numpy(depth.reshape(-1).copy()).to(DEV)
    ws = M.workspace(L, B, N)
    lg = torch.empty(R, shape.E, device=DEV)
    idx = torch.empty(R, shape.k, dtype=torch.int32, device=DEV)
    gates = torch.empty(R, shape.k, device=DEV)
    y = torch.empty(R, shape.d, dtype=torch.bfloat16, device=DEV)
    M.moe_tree_forward(L, P, x.to(DEV), wr, wg, wu, wd, None, dp, B, N, None, y, ws,
                       M.tree_outputs(logits=lg, topk_idx=idx, gates=gates),
                       M.run_opts(norm_input=True, residual=True))
    torch.cuda.synchronize()
    assert M.moe_workspace_check(ws) == 0
    xn = O.rmsnorm(x)
    ref_l = O.router(xn, wr.cpu())
    got_l = lg.cpu().numpy()
    assert (np.abs(got_l - ref_l) <= 1e-4 * np.abs(ref_l).max(axis=1, keepdims=True)).all()
    sel = O.select_block(got_l, depth, shape.k, W.C_EAGLE, mode=O.ACCEPT)
    np.testing.assert_array_equal(idx.cpu().numpy(), sel["idx"])
    np.testing.assert_allclose(gates.cpu().numpy(), sel["gates"], atol=1e-6)
    rows = sorted(np.random.default_rng(5).choice(R, 16, replace=False).tolist())
    moe = O.moe_combine(xn, wg.cpu(), wu.cpu(), wd.cpu(), sel["idx"], sel["gates"], rows=rows)
    ref = x.double().numpy()[rows] + moe
    got = y.double().cpu().numpy()[rows]
    assert np.abs(got - ref).max() <= 2e-2 * np.abs(ref).max()
    # the router sees the normalised rows: x and x / 4 (exact in bf16) give the same
    # logits up to the eps term and the roundings of the two normalised inputs
    lg1 = torch.empty_like(lg)
    x4 = (x / 4).to(DEV)
    M.moe_tree_forward(L, P, x4, wr, wg, wu, wd, None, dp, B, N, None, y, ws,
                       M.tree_outputs(logits=lg1), M.run_opts(norm_input=True))
    torch.cuda.synchronize()
    assert ((lg1 - lg).abs() <= 1e-3 * lg.abs().amax(1, keepdim=True)).all()


def test_normed_residual_chain_stays_bounded():
    """24 Qwen3-shaped layers (4 weight sets in turn) in a residual chain with the
    pre-norm, x <- x + MoE_l(norm(x)) stored in bf16: every layer's logits stay finite
    and O(1) (the norm keeps the router input at unit RMS) and the stream's RMS grows at
    most linearly in depth. Each layer is checked against the oracle on the device's
    own input to that layer: routing bit-exact from the device's logits and sampled rows
    of y within the bf16 bar."""
    shape = W.QWEN3_30B_A3B
    t = W.eagle_tree(61)
    N = t.N
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    sets = [_layer(shape, 70 + 3 * s, 0.1) for s in range(4)]
    x = W.hidden_states(62, t.parent, shape.d, torch.bfloat16).to(DEV)
    rms0 = x.double().pow(2).mean().sqrt().item()
    dep = torch.from_numpy(t.depth.copy()).to(DEV)
    ws = M.workspace(L, 1, N)
    lg = torch.empty(N, shape.E, device=DEV)
    idx = torch.empty(N, shape.k, dtype=torch.int32, device=DEV)
    rows = [0, 9, 33, 64]
    for layer in range(24):
        wr, wg, wu, wd = sets[layer % 4]
        x_in = x.clone()
        M.moe_tree_forward(L, P, x, wr, wg, wu, wd, None, dep, 1, N, None, x, ws,
                           M.tree_outputs(logits=lg, topk_idx=idx),
                           M.run_opts(norm_input=True, residual=True))
        torch.cuda.synchronize()
        got_l = lg.cpu().numpy()
        assert np.isfinite(got_l).all() and np.abs(got_l).max() < 50.0, layer
        if layer % 6 == 5:
            xi = x_in.cpu()
            sel = O.select_block(got_l, t.depth, shape.k, W.C_EAGLE, mode=O.ACCEPT)
            np.testing.assert_array_equal(idx.cpu().numpy(), sel["idx"])
            moe = O.moe_combine(O.rmsnorm(xi), wg.cpu(), wu.cpu(), wd.cpu(), sel["idx"],
                                sel["gates"], rows=rows)
            ref = xi.double().numpy()[rows] + moe
            got = x.double().cpu().numpy()[rows]
            assert np.abs(got - ref).max() <= 2e-2 * np.abs(ref).max(), layer
    assert torch.isfinite(x.float()).all()
    rms = x.double().pow(2).mean().sqrt().item()
    assert rms <= 25 * max(rms0, 1.0), (rms, rms0)


def test_normed_fp32_layer_against_oracle():
    """The fp32 layer (CUDA-core router and experts) with the pre-norm and the residual:
    routing bit-exact from the device's logits, every row of y within 1e-4 * max|ref|."""
    shape = W.TINY
    t = W.eagle_tree(81, steps=3, topk=4, draft_tokens=20)
    N = t.N
    x = (W.hidden_states(82, t.parent, shape.d, torch.float32) * 3.0)
    wr, wg, wu, wd = _layer(shape, 83, 0.3)
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "fp32")
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_TINY)
    dep = torch.from_numpy(t.depth.copy()).to(DEV)
    ws = M.workspace(L, 1, N)
    lg = torch.empty(N, shape.E, device=DEV)
    idx = torch.empty(N, shape.k, dtype=torch.int32, device=DEV)
    gates = torch.empty(N, shape.k, device=DEV)
    y = torch.empty(N, shape.d, device=DEV)
    M.moe_tree_forward(L, P, x.to(DEV), wr, wg, wu, wd, None, dep, 1, N, None, y, ws,
                       M.tree_outputs(logits=lg, topk_idx=idx, gates=gates),
                       M.run_opts(norm_input=True, residual=True))
    torch.cuda.synchronize()
    assert M.moe_workspace_check(ws) == 0
    xn = O.rmsnorm(x)
    ref_l = O.router(xn, wr.cpu())
    got_l = lg.cpu().numpy()
    assert (np.abs(got_l - ref_l) <= 1e-4 * np.abs(ref_l).max(axis=1, keepdims=True)).all()
    sel = O.select_tree(got_l, t.depth, shape.k, W.C_TINY, mode=O.ACCEPT)
    np.testing.assert_array_equal(idx.cpu().numpy(), sel["idx"])
    ref = x.double().numpy() + O.moe_combine(xn, wg.cpu(), wu.cpu(), wd.cpu(), sel["idx"],
                                             sel["gates"])
    got = y.double().cpu().numpy()
    assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max()
