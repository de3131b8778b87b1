"""Host-side checks of libmoetree that need no GPU: the library builds and loads,
exports every function include/moetree.h declares, rejects bad arguments before
touching CUDA, sizes workspaces, and runs the residency table's LRU logic."""
import os
import re

import numpy as np
import pytest

from expert_select_gb300 import build as B
from expert_select_gb300 import moetree as M

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert len(names) >= 16
    lib = M.lib()
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert names == set(M.EXPORTS)


def test_status_strings_and_version():
    assert M.status_str(0) == "ok"
    assert "slot" in M.status_str(M.MOE_ERR_NOSLOT)
    assert M.status_str(12345) == "unknown status"
    assert M.lib().moe_abi_version() == 202


def test_workspace_bytes():
    L = M.layer_desc(2048, 128, 8, 768, "bf16")
    n1 = M.moe_workspace_bytes(L, 1, 65)
    n64 = M.moe_workspace_bytes(L, 64, 65)
    assert 0 < n1 < n64 and n1 % 256 == 0
    assert M.moe_workspace_bytes(M.layer_desc(2048, 128, 0, 768, "bf16"), 1, 65) == 0
    assert M.moe_workspace_bytes(M.layer_desc(2047, 128, 8, 768, "bf16"), 1, 65) == 0
    assert M.moe_workspace_bytes(M.layer_desc(2048, 300, 8, 768, "bf16"), 1, 65) == 0
    assert M.moe_workspace_bytes(L, 0, 65) == 0


def test_bad_arguments_rejected_before_any_launch():
    import ctypes as C
    lib = M.lib()
    L = M.layer_desc(256, 16, 2, 128, "fp32")
    P = M.select_params(M.MOE_ROUTE_ACCEPT, [1.0, 0.5])
    nul = None
    assert lib.moe_router_logits(C.byref(L), nul, nul, 4, nul, nul) == M.MOE_ERR_ARG
    assert lib.moe_tree_select(C.byref(L), C.byref(P), nul, nul, 1, 9, nul, nul, nul, nul, nul,
                               nul) == M.MOE_ERR_ARG
    bad = M.select_params(7, [1.0])
    assert lib.moe_tree_select(C.byref(L), C.byref(bad), nul, nul, 0, 0, nul, nul, nul, nul, nul,
                               nul) == M.MOE_ERR_ARG
    Pp = M.select_params(M.MOE_ROUTE_ACCEPT, [1.0], prune=True)
    fake = C.c_void_p(256)  # never dereferenced: the missing residency mask fails first
    assert lib.moe_tree_select(C.byref(L), C.byref(Pp), fake, fake, 1, 9, nul, fake, fake, nul,
                               nul, nul) == M.MOE_ERR_ARG
    assert lib.moe_expert_forward(C.byref(L), nul, nul, nul, nul, nul, nul, nul, 9, nul, nul, nul,
                                  nul) == M.MOE_ERR_ARG
    assert lib.moe_tree_forward(C.byref(L), C.byref(P), nul, nul, nul, nul, nul, nul, nul, 1, 9,
                                nul, nul, nul, nul, nul, nul) == M.MOE_ERR_ARG
    # misaligned (not 16-byte) pointers are rejected on the host
    odd = C.c_void_p(0x1004)
    assert lib.moe_router_logits(C.byref(L), odd, odd, 4, odd, nul) == M.MOE_ERR_ARG
    assert lib.moe_rms_norm(C.byref(L), nul, 4, nul, nul) == M.MOE_ERR_ARG
    assert lib.moe_rms_norm(C.byref(L), odd, 4, odd, nul) == M.MOE_ERR_ARG
    assert lib.moe_rms_norm(C.byref(L), nul, -1, nul, nul) == M.MOE_ERR_ARG
    assert lib.moe_event_wait(nul, 1.0) == M.MOE_ERR_ARG


def test_draft_select_and_other_entry_points_reject_bad_arguments():
    import ctypes as C
    lib = M.lib()
    L = M.layer_desc(2048, 128, 8, 768, "bf16")
    f = C.c_void_p(0x100000)  # 16-byte aligned, never dereferenced: argument checks fail first
    nul = None

    def draft(Cn, lam, gamma, x=nul, xs=nul, parent=f):
        return lib.moe_draft_select(C.byref(L), Cn, parent, f, f, f, lam, gamma, x, f, f, f, xs,
                                    nul, nul)
    assert draft(4098, 0.1, 65) == M.MOE_ERR_ARG           # more candidates than supported
    assert draft(0, 0.1, 65) == M.MOE_ERR_ARG              # no candidates
    assert draft(411, -0.1, 65) == M.MOE_ERR_ARG           # negative cost weight
    assert draft(411, float("nan"), 65) == M.MOE_ERR_ARG   # NaN cost weight
    assert draft(411, 0.1, 0) == M.MOE_ERR_ARG             # nothing to select
    assert draft(411, 0.1, 65, x=f) == M.MOE_ERR_ARG       # x without x_sel
    assert draft(411, 0.1, 65, parent=nul) == M.MOE_ERR_ARG
    odd = C.c_void_p(0x100004)
    assert draft(411, 0.1, 65, x=odd, xs=f) == M.MOE_ERR_ARG  # rows not 16-byte aligned
    assert lib.moe_expert_permute(C.byref(L), f, 0, f, f, f, f, nul) == M.MOE_ERR_ARG
    assert lib.moe_tree_forward_noalloc(C.byref(L), nul, nul, nul, nul, nul, nul, nul, nul, 1, 65,
                                        nul, nul, nul, nul, nul) == M.MOE_ERR_ARG
    P = M.select_params(M.MOE_ROUTE_ACCEPT, [1.0])
    # router + selection from hidden states: missing outputs, misaligned x
    assert lib.moe_tree_route(C.byref(L), C.byref(P), f, f, f, 1, 65, nul, nul, f, f, nul, nul,
                              nul) == M.MOE_ERR_ARG
    assert lib.moe_tree_route(C.byref(L), C.byref(P), odd, f, f, 1, 65, nul, f, f, f, nul, nul,
                              nul) == M.MOE_ERR_ARG
    # block counters: no output struct, or neither arrays nor a workspace to read them from
    st = M.TreeStats()
    assert lib.moe_tree_block_stats(C.byref(L), 1, 65, f, f, nul, nul, nul) == M.MOE_ERR_ARG
    assert lib.moe_tree_block_stats(C.byref(L), 1, 65, nul, f, nul, C.byref(st),
                                    nul) == M.MOE_ERR_ARG
    assert lib.moe_tree_block_stats(C.byref(L), 0, 65, f, f, nul, C.byref(st),
                                    nul) == M.MOE_ERR_ARG
    assert lib.moe_noalloc_check(nul, nul) == M.MOE_ERR_ARG
    Ls = M.layer_desc(2048, 128, 8, 768, "bf16", slots=48)
    # no residency table
    assert lib.moe_offload_forward(C.byref(Ls), C.byref(P), f, f, f, f, f, f, f, f, nul, 0, f,
                                   1, 65, f, nul, nul, f, nul, nul, nul) == M.MOE_ERR_ARG


class _LruModel:
    """Independent model of the slot policy: hits refresh, misses take a free slot
    (lowest index) or evict the least recently used slot not needed now."""

    def __init__(self, slots):
        self.expert_in = [-1] * slots
        self.used = [0] * slots
        self.tick = 0

    def plan(self, needed):
        ups, hits = [], 0
        where = {e: s for s, e in enumerate(self.expert_in) if e >= 0}
        for e in needed:
            if e in where:
                self.tick += 1
                self.used[where[e]] = self.tick
                hits += 1
        for e in needed:
            if e in where:
                continue
            free = [s for s, x in enumerate(self.expert_in) if x < 0]
            if free:
                v = free[0]
            else:
                cands = [s for s, x in enumerate(self.expert_in) if x not in needed]
                v = min(cands, key=lambda s: (self.used[s], s))
                del where[self.expert_in[v]]
            self.expert_in[v] = e
            where[e] = v
            self.tick += 1
            self.used[v] = self.tick
            ups.append((e, v))
        return ups, hits


def test_residency_plan_follows_lru():
    E, slots = 32, 6
    R = M.Residency(n_layers=2, E=E, slots=slots)
    model = _LruModel(slots)
    rng = np.random.Generator(np.random.PCG64(3))
    for step in range(200):
        needed = rng.choice(E, size=int(rng.integers(0, slots + 1)), replace=False).tolist()
        ue, us, hits = R.plan(1, needed)
        ups, mh = model.plan(needed)
        assert list(zip(ue.tolist(), us.tolist())) == ups and hits == mh
        slot, res = R.query(1)
        for s, e in enumerate(model.expert_in):
            if e >= 0:
                assert slot[e] == s and res[e] == 1
        assert int(res.sum()) == sum(1 for e in model.expert_in if e >= 0)
    slot0, res0 = R.query(0)  # the other layer is untouched
    assert (slot0 == -1).all() and res0.sum() == 0


def test_residency_errors():
    R = M.Residency(n_layers=1, E=8, slots=3)
    assert R.upload_wait(0) == (0.0, 0)  # no offloaded call yet: no waits
    with pytest.raises(M.MoeError):
        R.upload_wait(1)
    with pytest.raises(M.MoeError) as ei:
        R.plan(0, [0, 1, 2, 3])
    assert ei.value.status == M.MOE_ERR_NOSLOT
    with pytest.raises(M.MoeError):
        R.plan(0, [1, 1])
    with pytest.raises(M.MoeError):
        R.plan(0, [9])
    with pytest.raises(M.MoeError):
        R.plan(3, [0])
    with pytest.raises(M.MoeError):
        M.Residency(n_layers=1, E=8, slots=9)
