"""Thin ctypes binding of libmoetree (include/moetree.h).

Argument marshalling only: every function takes torch tensors that already live
where the C ABI wants them (device or host), passes their data pointers, the
current CUDA stream and plain integers to the C entry point of the same name, and
raises MoeError on a non-zero status. All computation runs in the library's
kernels. The library is loaded from this package directory; if it is missing the
import of any entry point fails loudly (there is no fallback).
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoetree.so")

MOE_OK, MOE_ERR_ARG, MOE_ERR_CUDA, MOE_ERR_NOSLOT, MOE_ERR_TIMEOUT = 0, -1, -2, -3, -4
MOE_ERR_DEVICE_CHECK, MOE_ERR_UNSUPPORTED = -5, -6
MOE_DTYPE_F32, MOE_DTYPE_BF16 = 0, 1
MOE_ROUTE_NATURAL, MOE_ROUTE_ACCEPT, MOE_ROUTE_FIXED_B = 0, 1, 2
MOE_FFN_AUTO, MOE_FFN_SIMT, MOE_FFN_TCGEN05 = 0, 1, 2
MOE_MAX_DEPTHS = 16
MOE_INFO_FIELDS = 5

# Every function declared in include/moetree.h.
EXPORTS = (
    "moe_status_str", "moe_abi_version", "moe_workspace_bytes", "moe_router_logits",
    "moe_tree_select", "moe_expert_permute", "moe_expert_forward", "moe_tree_forward",
    "moe_workspace_check", "moe_residency_create", "moe_residency_destroy",
    "moe_residency_query", "moe_residency_plan", "moe_residency_publish", "moe_expert_upload",
    "moe_event_wait", "moe_tree_forward_noalloc", "moe_offload_forward", "moe_draft_select",
    "moe_tree_route", "moe_tree_block_stats", "moe_noalloc_check", "moe_offload_upload_wait",
    "moe_rms_norm",
)


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_str(status)} ({status})")
        self.status = status


class LayerDesc(C.Structure):
    _fields_ = [("d", C.c_int), ("E", C.c_int), ("k", C.c_int), ("f", C.c_int), ("dtype", C.c_int),
                ("slots", C.c_int)]


class SelectParams(C.Structure):
    _fields_ = [("mode", C.c_int), ("n_c", C.c_int), ("c_by_depth", C.c_double * MOE_MAX_DEPTHS),
                ("pool_all", C.c_int), ("anchor", C.c_int), ("prune", C.c_int),
                ("reroute_budget", C.c_int), ("min_set", C.c_int), ("fixed_B", C.c_int)]


class TreeOutputs(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in
                ("logits", "topk_idx", "gates", "eligible", "info", "counts", "offsets", "perm")]


class OffloadStats(C.Structure):
    _fields_ = [("needed", C.c_int), ("hits", C.c_int), ("uploads", C.c_int),
                ("passes", C.c_int), ("h2d_bytes", C.c_longlong)]


class TreeStats(C.Structure):
    _fields_ = [("trees", C.c_int), ("assignments", C.c_int), ("union_experts", C.c_int),
                ("max_per_expert", C.c_int), ("reuse", C.c_double),
                ("union_nat_mean", C.c_double), ("union_sel_mean", C.c_double),
                ("m_mean", C.c_double), ("pruned_mean", C.c_double), ("exact_trees", C.c_int)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class RunOpts(C.Structure):
    _fields_ = [("ffn_path", C.c_int), ("ffn_begin", C.c_void_p), ("ffn_end", C.c_void_p),
                ("residual", C.c_int), ("select_begin", C.c_void_p), ("norm_input", C.c_int),
                ("ffn_max_ctas", C.c_int)]


_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() "
                               "(the CUDA library is required; there is no fallback)")
        L = C.CDLL(LIB_PATH)
        P, I, S = C.c_void_p, C.c_int, C.c_size_t
        sig = {
            "moe_status_str": ([I], C.c_char_p),
            "moe_abi_version": ([], I),
            "moe_workspace_bytes": ([P, I, I], S),
            "moe_router_logits": ([P, P, P, I, P, P], I),
            "moe_rms_norm": ([P, P, I, P, P], I),
            "moe_tree_select": ([P, P, P, P, I, I, P, P, P, P, P, P], I),
            "moe_expert_permute": ([P, P, I, P, P, P, P, P], I),
            "moe_expert_forward": ([P, P, P, P, P, P, P, P, I, P, P, P, P], I),
            "moe_tree_forward": ([P, P, P, P, P, P, P, P, P, I, I, P, P, P, P, P, P], I),
            "moe_workspace_check": ([P, P, P], I),
            "moe_residency_create": ([I, I, I, P], I),
            "moe_residency_destroy": ([P], I),
            "moe_residency_query": ([P, I, P, P], I),
            "moe_residency_plan": ([P, I, P, I, P, P, P, P], I),
            "moe_residency_publish": ([P, I, P, P, P], I),
            "moe_expert_upload": ([P, P, P, P, P, P, P, P, P, I, P, P], I),
            "moe_event_wait": ([P, C.c_double], I),
            "moe_tree_forward_noalloc": ([P, P, P, P, P, P, P, P, P, I, I, P, P, P, P, P], I),
            "moe_offload_forward": ([P, P, P, P, P, P, P, P, P, P, P, I, P, I, I, P, P, P, P, P,
                                     P, P], I),
            "moe_draft_select": ([P, I, P, P, P, P, C.c_float, I, P, P, P, P, P, P, P], I),
            "moe_tree_route": ([P, P, P, P, P, I, I, P, P, P, P, P, P, P], I),
            "moe_tree_block_stats": ([P, I, I, P, P, P, P, P], I),
            "moe_noalloc_check": ([P, P], I),
            "moe_offload_upload_wait": ([P, I, C.c_double, P, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().moe_status_str(status).decode()


def _check(fn: str, status: int) -> int:
    if status != MOE_OK:
        raise MoeError(fn, status)
    return status


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def layer_desc(d: int, E: int, k: int, f: int, dtype, slots: int = 0) -> LayerDesc:
    """slots: expert slots in the weight pools (0 = E, one slot per expert)."""
    code = MOE_DTYPE_BF16 if dtype in (torch.bfloat16, "bf16") else MOE_DTYPE_F32
    return LayerDesc(d, E, k, f, code, slots)


def select_params(mode: int = MOE_ROUTE_ACCEPT, c: Sequence[float] = (1.0,), pool_all=False,
                  anchor=True, prune=False, reroute_budget=8, min_set=16, fixed_B=0) -> SelectParams:
    p = SelectParams()
    p.mode = mode
    p.n_c = len(c)
    for i, v in enumerate(c):
        p.c_by_depth[i] = float(v)
    p.pool_all, p.anchor, p.prune = int(pool_all), int(anchor), int(prune)
    p.reroute_budget, p.min_set, p.fixed_B = reroute_budget, min_set, fixed_B
    return p


def moe_workspace_bytes(L: LayerDesc, B: int, N: int) -> int:
    return int(lib().moe_workspace_bytes(C.byref(L), B, N))


def workspace(L: LayerDesc, B: int, N: int, device="cuda") -> torch.Tensor:
    """A device byte buffer of moe_workspace_bytes (torch allocations are 256-B aligned)."""
    n = moe_workspace_bytes(L, B, N)
    if n == 0:
        raise MoeError("moe_workspace_bytes", MOE_ERR_ARG)
    return torch.empty(n, dtype=torch.uint8, device=device)


def moe_router_logits(L, x, W_r, logits, stream=None):
    return _check("moe_router_logits", lib().moe_router_logits(
        C.byref(L), _ptr(x), _ptr(W_r), x.shape[0], _ptr(logits), _stream(stream)))


def moe_rms_norm(L, x, xn, stream=None):
    return _check("moe_rms_norm", lib().moe_rms_norm(
        C.byref(L), _ptr(x), x.shape[0], _ptr(xn), _stream(stream)))


def moe_tree_select(L, P, logits, depth, B, N, resident, topk_idx, gates, eligible=None,
                    info=None, stream=None):
    return _check("moe_tree_select", lib().moe_tree_select(
        C.byref(L), C.byref(P), _ptr(logits), _ptr(depth), B, N, _ptr(resident), _ptr(topk_idx),
        _ptr(gates), _ptr(eligible), _ptr(info), _stream(stream)))


def moe_tree_route(L, P, x, W_r, depth, B, N, resident, logits, topk_idx, gates, eligible=None,
                   info=None, stream=None):
    return _check("moe_tree_route", lib().moe_tree_route(
        C.byref(L), C.byref(P), _ptr(x), _ptr(W_r), _ptr(depth), B, N, _ptr(resident),
        _ptr(logits), _ptr(topk_idx), _ptr(gates), _ptr(eligible), _ptr(info), _stream(stream)))


def moe_tree_block_stats(L, B, N, info=None, counts=None, ws=None, stream=None) -> TreeStats:
    """Counters of the last block (union, reuse, per-tree set sizes); waits for the stream."""
    st = TreeStats()
    _check("moe_tree_block_stats", lib().moe_tree_block_stats(
        C.byref(L), B, N, _ptr(info), _ptr(counts), _ptr(ws), C.byref(st), _stream(stream)))
    return st


def moe_expert_permute(L, topk_idx, counts, offsets, perm, ws, stream=None):
    return _check("moe_expert_permute", lib().moe_expert_permute(
        C.byref(L), _ptr(topk_idx), topk_idx.shape[0], _ptr(counts), _ptr(offsets), _ptr(perm),
        _ptr(ws), _stream(stream)))


def _event(ev):
    if ev is None:
        return None
    if not ev.cuda_event:
        raise ValueError("torch.cuda.Event has no CUDA event yet: record it once first")
    return C.c_void_p(ev.cuda_event)


def run_opts(ffn_path: int = MOE_FFN_AUTO, begin=None, end=None, residual=False,
             select_begin=None, norm_input=False, ffn_max_ctas: int = 0) -> RunOpts:
    """Options for the forward entry points. `begin`/`end` are torch.cuda.Event
    objects recorded around the grouped-expert kernel, `select_begin` one recorded before
    the selection launch; `residual` returns x + MoE(x); `norm_input` routes and computes
    the experts on the RMS pre-norm of x (the residual still adds x); `ffn_max_ctas` caps
    the tensor-core expert kernel's CTAs (0: one per SM)."""
    return RunOpts(ffn_path, _event(begin), _event(end), int(residual), _event(select_begin),
                   int(norm_input), int(ffn_max_ctas))


def moe_expert_forward(L, x, W_gate, W_up, W_down, slot_of_expert, topk_idx, gates, y, ws,
                       opts: Optional[RunOpts] = None, stream=None):
    return _check("moe_expert_forward", lib().moe_expert_forward(
        C.byref(L), _ptr(x), _ptr(W_gate), _ptr(W_up), _ptr(W_down), _ptr(slot_of_expert),
        _ptr(topk_idx), _ptr(gates), x.shape[0], _ptr(y), _ptr(ws),
        None if opts is None else C.byref(opts), _stream(stream)))


def tree_outputs(**tensors) -> TreeOutputs:
    o = TreeOutputs()
    for k, v in tensors.items():
        setattr(o, k, None if v is None else v.data_ptr())
    return o


def moe_tree_forward(L, P, x, W_r, W_gate, W_up, W_down, slot_of_expert, depth, B, N, resident,
                     y, ws, out: Optional[TreeOutputs] = None, opts: Optional[RunOpts] = None,
                     stream=None):
    return _check("moe_tree_forward", lib().moe_tree_forward(
        C.byref(L), C.byref(P), _ptr(x), _ptr(W_r), _ptr(W_gate), _ptr(W_up), _ptr(W_down),
        _ptr(slot_of_expert), _ptr(depth), B, N, _ptr(resident), _ptr(y),
        None if out is None else C.byref(out), _ptr(ws),
        None if opts is None else C.byref(opts), _stream(stream)))


def moe_tree_forward_noalloc(L, P, x, W_r, W_gate, W_up, W_down, slot_of_expert, depth, B, N,
                             resident, y, out: Optional[TreeOutputs] = None,
                             opts: Optional[RunOpts] = None, stream=None):
    """moe_tree_forward with the library's built-in 16 MiB scratch instead of a
    caller-allocated workspace (for callers that cannot allocate device memory)."""
    return _check("moe_tree_forward_noalloc", lib().moe_tree_forward_noalloc(
        C.byref(L), C.byref(P), _ptr(x), _ptr(W_r), _ptr(W_gate), _ptr(W_up), _ptr(W_down),
        _ptr(slot_of_expert), _ptr(depth), B, N, _ptr(resident), _ptr(y),
        None if out is None else C.byref(out), None if opts is None else C.byref(opts),
        _stream(stream)))


def moe_workspace_check(ws, stream=None) -> int:
    flags = C.c_int(0)
    st = lib().moe_workspace_check(_ptr(ws), C.byref(flags), _stream(stream))
    if st not in (MOE_OK, MOE_ERR_DEVICE_CHECK):
        raise MoeError("moe_workspace_check", st)
    return flags.value


def moe_noalloc_check(stream=None) -> int:
    """Reads and clears the check word of moe_tree_forward_noalloc's built-in scratch."""
    flags = C.c_int(0)
    st = lib().moe_noalloc_check(C.byref(flags), _stream(stream))
    if st not in (MOE_OK, MOE_ERR_DEVICE_CHECK):
        raise MoeError("moe_noalloc_check", st)
    return flags.value


class Residency:
    """Owner of a moe_residency table (host metadata of the expert slots)."""

    def __init__(self, n_layers: int, E: int, slots: int):
        self.E, self.slots = E, slots
        h = C.c_void_p()
        _check("moe_residency_create", lib().moe_residency_create(n_layers, E, slots, C.byref(h)))
        self.h = h

    def close(self):
        if self.h:
            lib().moe_residency_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def query(self, layer: int):
        import numpy as np
        slot = np.empty(self.E, dtype=np.int32)
        res = np.empty(self.E, dtype=np.uint8)
        _check("moe_residency_query", lib().moe_residency_query(
            self.h, layer, slot.ctypes.data_as(C.c_void_p), res.ctypes.data_as(C.c_void_p)))
        return slot, res

    def plan(self, layer: int, needed):
        import numpy as np
        nd = np.ascontiguousarray(np.asarray(needed, dtype=np.int32))
        ue = np.empty(max(1, len(nd)), dtype=np.int32)
        us = np.empty(max(1, len(nd)), dtype=np.int32)
        n_up, hits = C.c_int(0), C.c_int(0)
        _check("moe_residency_plan", lib().moe_residency_plan(
            self.h, layer, nd.ctypes.data_as(C.c_void_p), len(nd), ue.ctypes.data_as(C.c_void_p),
            us.ctypes.data_as(C.c_void_p), C.byref(n_up), C.byref(hits)))
        return ue[:n_up.value].copy(), us[:n_up.value].copy(), hits.value

    def upload_wait(self, layer: int, timeout_s: float = 10.0):
        """(ms the compute stream waited for uploads, number of waits) in the last
        moe_offload_forward call on `layer`."""
        ms, n = C.c_double(0), C.c_int(0)
        _check("moe_offload_upload_wait", lib().moe_offload_upload_wait(
            self.h, layer, float(timeout_s), C.byref(ms), C.byref(n)))
        return ms.value, n.value

    def publish(self, layer: int, slot_dev=None, res_dev=None, stream=None):
        _check("moe_residency_publish", lib().moe_residency_publish(
            self.h, layer, _ptr(slot_dev), _ptr(res_dev), _stream(stream)))


def moe_expert_upload(L, host_gate, host_up, host_down, slot_gate, slot_up, slot_down,
                      up_expert, up_slot, side_stream, done_event=None):
    import numpy as np
    ue = np.ascontiguousarray(np.asarray(up_expert, dtype=np.int32))
    us = np.ascontiguousarray(np.asarray(up_slot, dtype=np.int32))
    return _check("moe_expert_upload", lib().moe_expert_upload(
        C.byref(L), _ptr(host_gate), _ptr(host_up), _ptr(host_down), _ptr(slot_gate),
        _ptr(slot_up), _ptr(slot_down), ue.ctypes.data_as(C.c_void_p),
        us.ctypes.data_as(C.c_void_p), len(ue), C.c_void_p(side_stream.cuda_stream),
        _event(done_event)))


def moe_offload_forward(L, P, x, W_r, host_gate, host_up, host_down, slot_gate, slot_up,
                        slot_down, table: "Residency", layer: int, depth, B, N, y, ws,
                        out: Optional[TreeOutputs] = None, opts: Optional[RunOpts] = None,
                        stream=None, side_stream=None) -> OffloadStats:
    """The layer with offloaded experts; returns the call's OffloadStats."""
    st = OffloadStats()
    side = side_stream if side_stream is not None else torch.cuda.current_stream()
    _check("moe_offload_forward", lib().moe_offload_forward(
        C.byref(L), C.byref(P), _ptr(x), _ptr(W_r), _ptr(host_gate), _ptr(host_up),
        _ptr(host_down), _ptr(slot_gate), _ptr(slot_up), _ptr(slot_down), table.h, layer,
        _ptr(depth), B, N, _ptr(y), None if out is None else C.byref(out), C.byref(st), _ptr(ws),
        None if opts is None else C.byref(opts), _stream(stream), C.c_void_p(side.cuda_stream)))
    return st


def moe_draft_select(L, parent, depth, logp, footprint, lam: float, gamma: int, selected,
                     sel_parent, sel_depth, x=None, x_sel=None, n_union=None, stream=None):
    """Cost-aware choice of the draft tree to verify (see include/moetree.h)."""
    return _check("moe_draft_select", lib().moe_draft_select(
        C.byref(L), parent.shape[0], _ptr(parent), _ptr(depth), _ptr(logp), _ptr(footprint),
        float(lam), gamma, _ptr(x), _ptr(selected), _ptr(sel_parent), _ptr(sel_depth),
        _ptr(x_sel), _ptr(n_union), _stream(stream)))


def moe_event_wait(event, timeout_s: float) -> None:
    _check("moe_event_wait", lib().moe_event_wait(_event(event), float(timeout_s)))
