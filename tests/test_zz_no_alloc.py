"""The allocation-free layer entry point, moe_tree_forward_noalloc.

Callers that cannot allocate device memory while they run (an engine whose free HBM
already belongs to its KV cache, a plug-in handed only input/output pointers, a
loop that must not let cudaMalloc synchronise the device) use this entry point; it
keeps its scratch in a built-in device array instead of a workspace argument.
This file is collected last so that a failure here stops a `-x` run only after
every other test has run; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from expert_select_gb300 import moetree as M
from expert_select_gb300 import workload as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def layer():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from expert_select_gb300 import build
    build.build()
    shape = W.QWEN3_30B_A3B
    wr = W.router_weight(901, shape, std=0.1, device=DEV)
    wg, wu, wd = W.expert_weights(902, shape, device=DEV)
    return shape, wr, wg, wu, wd


def _tree(seed, shape):
    t = W.eagle_tree(seed)
    x = W.hidden_states(seed + 1, t.parent, shape.d, shape.torch_dtype).to(DEV)
    return t, x, torch.from_numpy(t.depth.copy()).to(DEV)


def _outputs(shape, R):
    return dict(topk_idx=torch.empty(R, shape.k, dtype=torch.int32, device=DEV),
                counts=torch.empty(shape.E, dtype=torch.int32, device=DEV))


def test_noalloc_prenorm_residual_equals_workspace_forward(layer):
    """The pre-norm residual block (norm_input + residual, y written over x) through the
    built-in scratch equals the same call with a caller workspace bit for bit."""
    shape, wr, wg, wu, wd = layer
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    t, x, dep = _tree(31, shape)
    R = t.N
    opts = M.run_opts(residual=True, norm_input=True)
    y_ref = x.clone()
    y_na = x.clone()
    ws = M.workspace(L, 1, R)
    M.moe_tree_forward(L, P, y_ref, wr, wg, wu, wd, None, dep, 1, R, None, y_ref, ws, None, opts)
    M.moe_tree_forward_noalloc(L, P, y_na, wr, wg, wu, wd, None, dep, 1, R, None, y_na, None,
                               opts)
    torch.cuda.synchronize()
    assert M.moe_workspace_check(ws) == 0
    assert M.moe_noalloc_check() == 0
    assert torch.equal(y_na, y_ref)
    assert not torch.equal(y_na, x)


def test_noalloc_matches_workspace_forward_twice(layer):
    """Two calls in a row (different trees) through the built-in scratch give the
    same routing as moe_tree_forward with a caller workspace, and outputs within
    the layer tolerance max|dy| <= 2e-2 * max|y|."""
    shape, wr, wg, wu, wd = layer
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    for seed in (11, 12):
        t, x, dep = _tree(seed, shape)
        R = t.N
        ref_out, na_out = _outputs(shape, R), _outputs(shape, R)
        y_ref = torch.empty(R, shape.d, dtype=torch.bfloat16, device=DEV)
        y_na = torch.full((R, shape.d), float("nan"), dtype=torch.bfloat16, device=DEV)
        ws = M.workspace(L, 1, R)
        M.moe_tree_forward(L, P, x, wr, wg, wu, wd, None, dep, 1, R, None, y_ref, ws,
                           M.tree_outputs(**ref_out))
        M.moe_tree_forward_noalloc(L, P, x, wr, wg, wu, wd, None, dep, 1, R, None, y_na,
                                   M.tree_outputs(**na_out))
        torch.cuda.synchronize()
        assert torch.equal(ref_out["topk_idx"], na_out["topk_idx"])
        assert torch.equal(ref_out["counts"], na_out["counts"])
        a, b = y_ref.float().cpu().numpy(), y_na.float().cpu().numpy()
        assert np.isfinite(b).all()
        assert np.abs(a - b).max() <= 2e-2 * np.abs(a).max()


def test_noalloc_rejects_requests_beyond_its_scratch(layer):
    shape, wr, wg, wu, wd = layer
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    B, N = 4, 65  # about 31 MiB of scratch: more than the built-in 16 MiB
    assert M.moe_workspace_bytes(L, B, N) > 16 << 20
    x = torch.zeros(B * N, shape.d, dtype=torch.bfloat16, device=DEV)
    dep = torch.zeros(B * N, dtype=torch.int32, device=DEV)
    y = torch.empty_like(x)
    with pytest.raises(M.MoeError) as ei:
        M.moe_tree_forward_noalloc(L, P, x, wr, wg, wu, wd, None, dep, B, N, None, y)
    assert ei.value.status == M.MOE_ERR_UNSUPPORTED


def test_noalloc_reports_kernel_checks(layer):
    """The built-in scratch's check word is readable (and cleared) through
    moe_noalloc_check: an expert mapped to a slot outside the weight pool is skipped by
    the expert kernel and flagged (bit 0); a clean call reports 0."""
    shape, wr, wg, wu, wd = layer
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    t, x, dep = _tree(13, shape)
    R = t.N
    y = torch.empty(R, shape.d, dtype=torch.bfloat16, device=DEV)
    M.moe_tree_forward_noalloc(L, P, x, wr, wg, wu, wd, None, dep, 1, R, None, y)
    assert M.moe_noalloc_check() == 0
    slot = torch.arange(shape.E, dtype=torch.int32, device=DEV)
    idx = torch.empty(R, shape.k, dtype=torch.int32, device=DEV)
    M.moe_tree_forward_noalloc(L, P, x, wr, wg, wu, wd, slot, dep, 1, R, None, y,
                               M.tree_outputs(topk_idx=idx))
    torch.cuda.synchronize()
    slot[int(idx[0, 0].item())] = 10 ** 6  # the root's first expert: beyond the pool
    M.moe_tree_forward_noalloc(L, P, x, wr, wg, wu, wd, slot, dep, 1, R, None, y)
    assert M.moe_noalloc_check() & 1
    assert M.moe_noalloc_check() == 0  # cleared by the read
