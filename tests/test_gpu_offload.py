"""GPU tests of the offloaded layer (moe_offload_forward) and of the residual option.

The offloaded layer computes every expert with the same kernels as the resident layer
(with or without the pre-norm and the residual),
only addressed through slots that uploads fill, in one or more passes; so its output
must equal moe_tree_forward on the same inputs bit for bit, given the residency mask the
table had before the call (pruning reads that mask). The counters must add up: every
needed expert is either a hit or uploaded once, and the bytes copied are the uploaded
experts' weights.
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


SHAPE_TC = W.LayerShape(d=256, E=32, k=4, f=128, dtype="bf16")
SHAPE_SIMT = W.LayerShape(d=256, E=16, k=2, f=128, dtype="fp32")


def _params(mode, prune):
    if mode == "natural":
        return M.select_params(M.MOE_ROUTE_NATURAL, W.C_EAGLE)
    return M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE, prune=prune, reroute_budget=8,
                           min_set=4)


@pytest.mark.parametrize("shape,slots,mode,prune,router_std,norm", [
    (SHAPE_TC, 8, "natural", False, 0.02, False),
    (SHAPE_TC, 8, "accept", False, 0.3, False),
    (SHAPE_TC, 12, "accept", True, 0.3, False),
    (SHAPE_TC, 12, "accept", True, 0.3, True),
    (SHAPE_TC, 30, "natural", False, 0.02, False),
    (SHAPE_SIMT, 4, "accept", True, 0.3, False),
    (SHAPE_SIMT, 4, "accept", True, 0.3, True),
])
def test_offload_matches_resident_layer(shape, slots, mode, prune, router_std, norm):
    E, k = shape.E, shape.k
    wg, wu, wd = W.expert_weights(5, shape, device=DEV)
    hg, hu, hd = (w.cpu().pin_memory() for w in (wg, wu, wd))
    pg = torch.zeros(slots, shape.f, shape.d, dtype=shape.torch_dtype, device=DEV)
    pu = torch.zeros_like(pg)
    pd = torch.zeros(slots, shape.d, shape.f, dtype=shape.torch_dtype, device=DEV)
    wr = W.router_weight(6, shape, std=router_std, device=DEV)
    L = M.layer_desc(shape.d, E, k, shape.f, shape.dtype)
    Ls = M.layer_desc(shape.d, E, k, shape.f, shape.dtype, slots=slots)
    P = _params(mode, prune)
    table = M.Residency(n_layers=2, E=E, slots=slots)
    side = torch.cuda.Stream()
    expert_bytes = 3 * shape.d * shape.f * shape.elem_bytes
    total_up = 0
    for step in range(4):
        t = W.eagle_tree(40 + step)
        N = t.N
        x = W.hidden_states(50 + step, t.parent, shape.d, shape.torch_dtype).to(DEV)
        dep = torch.from_numpy(t.depth.copy()).to(DEV)
        _, res_before = table.query(1)
        res_dev = torch.from_numpy(res_before.copy()).to(DEV)
        # the resident layer, pruning against the same residency
        idx_ref = torch.empty(N, k, dtype=torch.int32, device=DEV)
        cnt_ref = torch.empty(E, dtype=torch.int32, device=DEV)
        y_ref = torch.empty(N, shape.d, dtype=shape.torch_dtype, device=DEV)
        ws = M.workspace(L, 1, N)
        opts = M.run_opts(norm_input=norm, residual=norm)
        M.moe_tree_forward(L, P, x, wr, wg, wu, wd, None, dep, 1, N, res_dev, y_ref, ws,
                           M.tree_outputs(topk_idx=idx_ref, counts=cnt_ref), opts)
        # the offloaded layer
        idx = torch.empty_like(idx_ref)
        y = torch.full_like(y_ref, float("nan"))
        ws2 = M.workspace(Ls, 1, N)
        st = M.moe_offload_forward(Ls, P, x, wr, hg, hu, hd, pg, pu, pd, table, 1, dep, 1, N,
                                   y, ws2, M.tree_outputs(topk_idx=idx), opts=opts,
                                   side_stream=side)
        torch.cuda.synchronize()
        assert M.moe_workspace_check(ws2) == 0
        assert torch.equal(idx, idx_ref)
        assert torch.equal(y, y_ref), step
        union = int((cnt_ref > 0).sum())
        assert st.needed == union
        assert st.hits + st.uploads == union
        assert st.h2d_bytes == st.uploads * expert_bytes
        if union > slots:
            assert st.passes >= 2
        # one timed wait per pass that needed uploads; a wait lasts >= 0 ms
        wait_ms, waits = table.upload_wait(1)
        assert waits == st.passes - (1 if st.hits > 0 else 0)
        assert wait_ms >= 0.0 and (waits > 0 or wait_ms == 0.0)
        total_up += st.uploads
        slot_map, res_after = table.query(1)
        needed = np.flatnonzero(cnt_ref.cpu().numpy())
        # the last pass's experts are resident; at most `slots` experts are
        assert int(res_after.sum()) <= slots
        assert len(set(slot_map[slot_map >= 0].tolist())) == int(res_after.sum())
        if union <= slots:
            assert res_after[needed].all()
    assert total_up > 0


def test_residual_option_adds_the_input():
    shape = W.QWEN3_30B_A3B
    t = W.eagle_tree(3)
    N = t.N
    x = W.hidden_states(4, t.parent, shape.d, torch.bfloat16).to(DEV)
    dep = torch.from_numpy(t.depth.copy()).to(DEV)
    wr = W.router_weight(7, shape, std=0.1, device=DEV)
    wg, wu, wd = W.expert_weights(8, shape, device=DEV)
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE)
    ws = M.workspace(L, 1, N)
    y = torch.empty_like(x)
    M.moe_tree_forward(L, P, x, wr, wg, wu, wd, None, dep, 1, N, None, y, ws)
    yr = x.clone()  # in place: y aliases x
    M.moe_tree_forward(L, P, yr, wr, wg, wu, wd, None, dep, 1, N, None, yr, ws, None,
                       M.run_opts(residual=True))
    torch.cuda.synchronize()
    ref = x.double() + y.double()
    err = (yr.double() - ref).abs().max().item()
    assert err <= 2e-2 * ref.abs().max().item()


def test_offload_gptoss_shape_against_oracle():
    """A GPT-OSS-120B-shaped offloaded layer (d = f = 2880, top-4, bf16; 32 experts, 12
    slots, AcceptMoE with residency-aware pruning, router std 0.1), two blocks in a row:
    the routing equals the fp64 oracle's on the device's logits and the residency the
    table had before each call, and sampled rows of y equal the oracle's experts and
    combine within the bf16 bar."""
    shape = W.LayerShape(d=2880, E=32, k=4, f=2880, dtype="bf16")
    slots = 12
    wg, wu, wd = W.expert_weights(15, shape, device=DEV)
    hg, hu, hd = (w.cpu().pin_memory() for w in (wg, wu, wd))
    del wg, wu, wd
    pg = torch.zeros(slots, shape.f, shape.d, dtype=torch.bfloat16, device=DEV)
    pu = torch.zeros_like(pg)
    pd = torch.zeros(slots, shape.d, shape.f, dtype=torch.bfloat16, device=DEV)
    wr = W.router_weight(16, shape, std=0.1, device=DEV)
    Ls = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16", slots=slots)
    P = M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE, prune=True, reroute_budget=8, min_set=4)
    table = M.Residency(n_layers=1, E=shape.E, slots=slots)
    side = torch.cuda.Stream()
    for step in range(2):
        t = W.eagle_tree(70 + step)
        N = t.N
        x = W.hidden_states(80 + step, t.parent, shape.d, torch.bfloat16).to(DEV)
        dep = torch.from_numpy(t.depth.copy()).to(DEV)
        _, res_before = table.query(0)
        lg = torch.empty(N, shape.E, device=DEV)
        idx = torch.empty(N, shape.k, dtype=torch.int32, device=DEV)
        g = torch.empty(N, shape.k, device=DEV)
        y = torch.empty(N, shape.d, dtype=torch.bfloat16, device=DEV)
        ws = M.workspace(Ls, 1, N)
        st = M.moe_offload_forward(Ls, P, x, wr, hg, hu, hd, pg, pu, pd, table, 0, dep, 1, N, y,
                                   ws, M.tree_outputs(logits=lg, topk_idx=idx, gates=g),
                                   side_stream=side)
        torch.cuda.synchronize()
        assert M.moe_workspace_check(ws) == 0
        assert st.uploads > 0 and st.hits + st.uploads == st.needed
        sel = O.select_tree(lg.cpu().numpy(), t.depth, shape.k, W.C_EAGLE, mode=O.ACCEPT,
                            prune=True, resident=res_before, budget=8, min_set=4)
        np.testing.assert_array_equal(idx.cpu().numpy(), sel["idx"])
        rows = [0, 17, 40, 64]
        ref = O.moe_combine(x.cpu(), hg, hu, hd, sel["idx"], sel["gates"], rows=rows)
        got = y.float().cpu().numpy()[rows]
        assert np.abs(got - ref).max() <= 2e-2 * np.abs(ref).max()
