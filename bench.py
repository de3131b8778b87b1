"""Benchmark: the MoE tree-verification layer (Qwen3-30B-A3B-shaped, resident).

One step = one pass of the whole hot path over one verification block: router,
natural top-k, AcceptMoE selection (demand, effective-rank size, root anchor,
fill), restricted top-k, permute, grouped SwiGLU experts over the union, and the
gated combine, through the C entry point moe_tree_forward. Each step verifies a
different seeded EAGLE-3-shaped draft tree (65 nodes). Throughput is verification
blocks per second; the grouped-expert kernel is also reported against the HBM
roofline on its algorithmic bytes (union expert weights + token rows in/out).

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

With N > 1 (launched by torch.distributed.run) every rank runs an independent
replica on its own GPU (the layer has no cross-GPU exchange); the reported value is
the blocks all ranks processed divided by the slowest rank's time.

--impl reference times the CPU oracle instead (the checker): whole trees of the same
workload, spread over the host's cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE verify layer tree-blocks/s; union expert-weight HBM GB/s vs ~8 TB/s"
UNIT = "tree-blocks/s"
TREES = 64            # distinct seeded trees cycled through by the steps
REF_MAX_TREES = 320   # reference arm: whole trees timed at most (the rest of K is not run)
REF_MAX_WARMUP = 16   # reference arm: warm-up trees at most
SEED = 1000           # seed base of this workload


def workload_config(shape, routing, router_std):
    return {"workload": "qwen3-30b-a3b-moe-layer-resident-eagle3-tree",
            "d": shape.d, "E": shape.E, "k": shape.k, "f": shape.f,
            "tree_nodes": 65, "trees_per_block": 1, "draft": "eagle3 5 steps top-10 64 tokens",
            "routing": routing, "router_std": router_std, "commitment": "1,.8,.55,.35,.2,.1",
            "l2": "inputs larger than L2: each step streams ~0.7 GB of union expert weights "
                  "(L2 is 126 MB)"}


# ----------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Max of a per-rank float over the process group (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(units_per_rank: int, world: int, slowest_s: float) -> float:
    return units_per_rank * world / slowest_s


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                f = [v.strip() for v in line.split(",")]
                if len(f) >= 9 and f[1].replace(".", "").isdigit():
                    rows.append(f)
        except OSError:
            pass
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit()),
                "reasons": reasons, "samples": len(rows)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_sha(names=("ffn_tc.cu", "tc.cuh")):
    """sha256 (16 hex digits) of the expert kernel's sources, concatenated in order."""
    import hashlib
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "expert_select_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(mean_union: float):
    """DRAM bytes (read + write) per launch of the expert kernel, from the ncu capture
    summarised in profiles/ (bytes per union expert x this run's mean union), or None
    when that capture was taken on a different version of the kernel source."""
    path = os.path.join(ROOT, "profiles", "ffn_tcgen05_qwen3_layer.md")
    try:
        for line in open(path):
            if line.startswith("traffic_bytes_per_union_expert:"):
                f = line.split()
                if f[3] == kernel_sha():
                    return int(float(f[1]) * mean_union)
    except (OSError, IndexError, ValueError):
        pass
    return None


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# --------------------------------------------------------------- workload

def make_trees(n_trees: int, shape, seed: int):
    import torch
    from expert_select_gb300 import workload as W
    xs, deps = [], []
    for i in range(n_trees):
        t = W.eagle_tree(seed + i)
        xs.append(W.hidden_states(seed + 10_000 + i, t.parent, shape.d, shape.torch_dtype))
        deps.append(torch.from_numpy(t.depth.copy()))
    return torch.stack(xs), torch.stack(deps)


def oracle_block(x, wr, wg, wu, wd, depth, shape, routing, rows=None):
    """The oracle on one tree (optionally only `rows` of its expert outputs)."""
    from expert_select_gb300 import workload as W
    from oracle import oracle as O
    mode = O.ACCEPT if routing == "acceptmoe" else O.NATURAL
    return O.forward(x, wr, wg, wu, wd, depth, shape.k, W.C_EAGLE, rows=rows, mode=mode)


def time_oracle(xs, deps, wr, wg, wu, wd, shape, routing, n_trees):
    """Seconds per tree-block of the oracle on whole trees (all rows), one core."""
    per = []
    for i in range(n_trees):
        t0 = time.perf_counter()
        oracle_block(xs[i % len(xs)], wr, wg, wu, wd, deps[i % len(deps)].numpy(), shape,
                     routing)
        per.append(time.perf_counter() - t0)
    return per


_ORACLE_JOB = None


def _oracle_worker_init(xs, deps, wr, wg, wu, wd, shape, routing):
    """Runs in each spawned worker: keeps the (shared-memory) inputs of the workload."""
    os.environ["OMP_NUM_THREADS"] = "1"
    global _ORACLE_JOB
    _ORACLE_JOB = (xs, deps, wr, wg, wu, wd, shape, routing)
    from oracle import oracle as O
    O.lib()


def _oracle_worker_tree(i):
    xs, deps, wr, wg, wu, wd, shape, routing = _ORACLE_JOB
    t0 = time.perf_counter()
    oracle_block(xs[i % len(xs)], wr, wg, wu, wd, deps[i % len(deps)].numpy(), shape, routing)
    return time.perf_counter() - t0


class OraclePool:
    """The oracle on whole trees, one tree per task, over `procs` worker processes (spawned,
    never forked: the parent may hold a CUDA context). The inputs go to the workers once, as
    shared-memory tensors."""

    def __init__(self, procs, xs, deps, wr, wg, wu, wd, shape, routing):
        import torch.multiprocessing as mp
        for t in (xs, deps, wr, wg, wu, wd):
            t.share_memory_()
        self.procs = procs
        self.pool = mp.get_context("spawn").Pool(
            procs, initializer=_oracle_worker_init,
            initargs=(xs, deps, wr, wg, wu, wd, shape, routing))
        self.pool.map(_oracle_worker_tree, range(procs))  # imports and first calls, untimed

    def run(self, first, n):
        """Wall seconds to run trees first .. first + n - 1, and each tree's own seconds."""
        t0 = time.perf_counter()
        per = self.pool.map(_oracle_worker_tree, range(first, first + n), chunksize=1)
        return time.perf_counter() - t0, per

    def close(self):
        self.pool.close()
        self.pool.join()


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ------------------------------------------------------------------ GPU arm

def run_gpu(args):
    import torch
    from expert_select_gb300 import build
    from expert_select_gb300 import moetree as M
    from expert_select_gb300 import workload as W

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()

    shape = W.QWEN3_30B_A3B
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    seed = SEED + 7919 * rank
    xs_h, deps_h = make_trees(TREES, shape, seed)
    wr_std = args.router_std
    wr = W.router_weight(seed + 1, shape, std=wr_std, device=dev)
    wg, wu, wd = W.expert_weights(seed + 2, shape, device=dev)
    xs = xs_h.to(dev)
    deps = deps_h.to(dev).int()
    N = xs.shape[1]
    ws = M.workspace(L, 1, N, device=dev)
    y = torch.empty(N, shape.d, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.current_stream(dev)
    routing_mode = {"acceptmoe": M.MOE_ROUTE_ACCEPT, "natural": M.MOE_ROUTE_NATURAL}
    K, Wm = args.steps, args.warmup
    routing = args.routing
    other = "natural" if routing != "natural" else "acceptmoe"

    def loop(n, routing, w_r=wr, counts=None, info=None, ev=None):
        """n steps of the layer; with counts/info the step also writes its counters, with
        ev it records events around the expert stage (separate passes: both add work or
        launch gaps that the headline loop must not carry)."""
        P = M.select_params(routing_mode[routing], W.C_EAGLE)
        opts = M.run_opts(args.ffn_path)
        for i in range(n):
            j = i % TREES
            out = None
            if counts is not None:
                out = M.tree_outputs(counts=counts[i], info=info[i])
            if ev is not None:
                opts = M.run_opts(args.ffn_path, ev[i][1], ev[i][2], select_begin=ev[i][0])
            M.moe_tree_forward(L, P, xs[j], w_r, wg, wu, wd, None, deps[j], 1, N, None, y, ws,
                               out, opts)

    def runner(n, routing, w_r=wr):
        """A callable running n steps of the layer: by default CUDA graphs of the steps,
        captured here after the eager warm-up (the host then launches one graph instead of
        five kernels per step, and the programmatic launch edges between consecutive
        kernels stay inside the graph); with --no-graph the eager loop. Graphs hold up to
        256 steps (a multiple of the 64 trees, so replays walk the same tree sequence)."""
        if args.no_graph:
            return lambda: loop(n, routing, w_r=w_r)
        full, rest = divmod(n, 256)
        graphs = []
        for m in ([256] if full else []) + ([rest] if rest else []):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                loop(m, routing, w_r=w_r)
            graphs.append(g)
        torch.cuda.synchronize(dev)

        def run():
            for _ in range(full):
                graphs[0].replay()
            if rest:
                graphs[-1].replay()
        run()  # one untimed replay: the graphs' own first launch
        torch.cuda.synchronize(dev)
        return run

    def timed(n, routing, **kw):
        return _timed(runner(n, routing, **kw), dev, world)

    def counters(n, routing, **kw):
        """Per-step union (experts with assignments) and per-tree counters of the first n
        steps (the same trees as the timed loop), computed in an untimed pass."""
        counts = torch.zeros(n, shape.E, dtype=torch.int32, device=dev)
        info = torch.zeros(n, M.MOE_INFO_FIELDS, dtype=torch.int32, device=dev)
        loop(n, routing, counts=counts, info=info, **kw)
        torch.cuda.synchronize(dev)
        return (counts.cpu().numpy() > 0).sum(axis=1), info.cpu().numpy()

    # 1. the headline: K steps of the layer and nothing else in the timed region
    loop(Wm, routing)
    with ClockSampler(local) as clk:
        sec = timed(K, routing)
    clocks = clk.summary()
    value = whole_job_rate(K, world, sec)

    # 2. counters of the same steps (untimed pass)
    union, inf = counters(K, routing)
    assignments = N * shape.k

    # 3. the roofline window: events on every step of a separate pass, from just before
    # the selection launch (whose extra CTAs prefetch the root's experts into L2) to the
    # end of the grouped-expert kernel, and around the expert kernel alone
    K_ev = min(K, 1024)
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(K_ev)]
    for e3 in ev:  # torch creates the CUDA event on first record
        for e in e3:
            e.record(s)
    torch.cuda.synchronize(dev)
    loop(K_ev, routing, ev=ev)
    torch.cuda.synchronize(dev)
    stage_ms = np.array([a.elapsed_time(c) for a, _, c in ev])
    ffn_ms = np.array([b_.elapsed_time(c) for _, b_, c in ev])
    u_ev = union[np.arange(K_ev) % len(union)] if K_ev > K else union[:K_ev]
    stage_bytes = u_ev * shape.expert_bytes + 2 * N * shape.d * shape.elem_bytes
    peak, peak_kind = measured_peaks()
    achieved = float(stage_bytes.sum() / (stage_ms.sum() / 1e3)) / 1e9
    ffn_only = float(stage_bytes.sum() / (ffn_ms.sum() / 1e3)) / 1e9
    # whole step: the per-block algorithmic bytes of the layer (union expert weights, router
    # weights, token rows, SwiGLU activations) over the headline's time per step
    step_bytes = (union * shape.expert_bytes + shape.E * shape.d * shape.elem_bytes +
                  3 * N * shape.d * shape.elem_bytes + 2 * assignments * shape.f * 2)
    whole = float(step_bytes.mean() / (sec / K)) / 1e9
    traffic = measured_traffic(float(union.mean()))

    # end to end through the C ABI with host buffers (pinned), copies inside the timed
    # region: a copy stream brings step i+1's inputs in while step i computes and takes
    # step i's result out once it is done (double-buffered device inputs and outputs)
    xh = xs_h.pin_memory()
    dh = deps_h.int().pin_memory()
    yh = torch.empty(TREES, N, shape.d, dtype=torch.bfloat16).pin_memory()
    xin = [torch.empty_like(xs[0]) for _ in range(2)]
    din = [torch.empty_like(deps[0]) for _ in range(2)]
    yout = [torch.empty_like(y) for _ in range(2)]
    cs = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]

    def e2e_loop(n):
        P = M.select_params(routing_mode[routing], W.C_EAGLE)
        with torch.cuda.stream(cs):
            xin[0].copy_(xh[0], non_blocking=True)
            din[0].copy_(dh[0], non_blocking=True)
            ev_in[0].record(cs)
        for i in range(n):
            b, nb = i % 2, (i + 1) % 2
            if i + 1 < n:
                with torch.cuda.stream(cs):
                    if i >= 1:
                        cs.wait_event(ev_out[nb])  # step i-1 is done reading slot nb
                    xin[nb].copy_(xh[(i + 1) % TREES], non_blocking=True)
                    din[nb].copy_(dh[(i + 1) % TREES], non_blocking=True)
                    ev_in[nb].record(cs)
            s.wait_event(ev_in[b])
            if i >= 2:
                s.wait_event(ev_free[b])  # step i-2's result has left slot b
            M.moe_tree_forward(L, P, xin[b], wr, wg, wu, wd, None, din[b], 1, N, None, yout[b],
                               ws, None, M.run_opts(args.ffn_path))
            ev_out[b].record(s)
            with torch.cuda.stream(cs):
                cs.wait_event(ev_out[b])
                yh[i % TREES].copy_(yout[b], non_blocking=True)
                ev_free[b].record(cs)
        s.wait_event(ev_free[(n - 1) % 2])

    e2e_loop(Wm)
    torch.cuda.synchronize(dev)
    sec_e2e = _timed(lambda: e2e_loop(K), dev, world)
    e2e = {"value": whole_job_rate(K, world, sec_e2e), "unit": UNIT,
           "h2d_bytes_per_step": int(xin[0].numel() * xin[0].element_size() + din[0].numel() * 4),
           "d2h_bytes_per_step": int(yout[0].numel() * yout[0].element_size()),
           "pipelining": "copy stream: next step's inputs in, this step's output out"}

    # the other routing on the same trees (the pages' Standard SD), and both routings with
    # a peaked router (std 0.1, set sizes in the pages' 23-34 range), where selection
    # shrinks the union
    Kv = min(K, 2000)
    loop(Wm, other)
    sec_o = timed(Kv, other)
    u_o, _ = counters(Kv, other)
    wr_peaked = W.router_weight(seed + 1, shape, std=0.1, device=dev)
    peaked = {}
    for r_ in ("acceptmoe", "natural"):
        loop(Wm, r_, w_r=wr_peaked)
        sec_p = timed(Kv, r_, w_r=wr_peaked)
        u_p, i_p = counters(Kv, r_, w_r=wr_peaked)
        peaked[r_] = {"value": round(whole_job_rate(Kv, world, sec_p), 2),
                      "union_mean": round(float(u_p.mean()), 2),
                      "m_mean": round(float(i_p[:, 2].mean()), 2),
                      "reuse_mean": round(float(1 - u_p.mean() / assignments), 4),
                      "whole_step_hbm_frac": round(float(
                          (u_p * shape.expert_bytes + shape.E * shape.d * 2 +
                           3 * N * shape.d * 2 + 2 * assignments * shape.f * 2).mean()
                          / (sec_p / Kv) / 1e9 / peak), 4)}
    peaked["acceptmoe_vs_natural"] = round(peaked["acceptmoe"]["value"] /
                                           peaked["natural"]["value"], 3)

    # two independent one-tree blocks in flight (a serving engine verifying two requests'
    # trees at once): the trees alternate between two streams with their own workspaces,
    # and the expert kernel is capped below one CTA per SM so that one stream's routing
    # kernels find SMs while the other's experts stream. Reported beside the headline, not
    # instead of it: each call is still the one-tree layer.
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    cap = max(1, nsm - args.pair_free_sms)
    s2 = torch.cuda.Stream(dev)
    ws2 = M.workspace(L, 1, N, device=dev)
    y2 = torch.empty_like(y)

    def pair_loop(n, routing, w_r):
        P = M.select_params(routing_mode[routing], W.C_EAGLE)
        opts = M.run_opts(args.ffn_path, ffn_max_ctas=cap)
        cur = torch.cuda.current_stream(dev)
        s2.wait_stream(cur)
        for i in range(n):
            j = i % TREES
            if i % 2 == 0:
                M.moe_tree_forward(L, P, xs[j], w_r, wg, wu, wd, None, deps[j], 1, N, None, y,
                                   ws, None, opts, cur)
            else:
                M.moe_tree_forward(L, P, xs[j], w_r, wg, wu, wd, None, deps[j], 1, N, None, y2,
                                   ws2, None, opts, s2)
        cur.wait_stream(s2)

    def pair_runner(n, routing, w_r):
        if args.no_graph:
            return lambda: pair_loop(n, routing, w_r)
        full, rest = divmod(n, 256)
        graphs = []
        for m_ in ([256] if full else []) + ([rest] if rest else []):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                pair_loop(m_, routing, w_r)
            graphs.append(g)
        torch.cuda.synchronize(dev)

        def run():
            for _ in range(full):
                graphs[0].replay()
            if rest:
                graphs[-1].replay()
        run()
        torch.cuda.synchronize(dev)
        return run

    pair = {"ffn_ctas": cap, "streams": 2}
    for label, r_, w_r, u_ref in ((f"{routing}_std_{args.router_std:g}", routing, wr, union),
                                  ("acceptmoe_std_0.1", "acceptmoe", wr_peaked, None),
                                  ("natural_std_0.1", "natural", wr_peaked, None)):
        pair_loop(Wm, r_, w_r)
        torch.cuda.synchronize(dev)
        sec_pair = _timed(pair_runner(Kv, r_, w_r), dev, world)
        u_pair = u_ref[:Kv] if u_ref is not None else counters(Kv, r_, w_r=w_r)[0]
        pb = (u_pair * shape.expert_bytes + shape.E * shape.d * 2 + 3 * N * shape.d * 2 +
              2 * assignments * shape.f * 2).mean()
        pair[label] = {"value": round(whole_job_rate(Kv, world, sec_pair), 2),
                       "union_mean": round(float(u_pair.mean()), 2),
                       "whole_step_hbm_frac": round(float(pb / (sec_pair / Kv) / 1e9 / peak), 4)}

    # router, select, combine + the grouped-expert launches; the permute step runs inside
    # the selection launch for a block of one tree of up to 256 nodes, else in its own
    # kernel (and a second, placing kernel past 2048 assignments)
    permute_launches = 0 if N <= 256 else (2 if N * shape.k > 2048 else 1)
    launches_per_step = 3 + permute_launches + ffn_launches(M, L, args.ffn_path)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        wr_h, wg_h, wu_h, wd_h = wr.cpu(), wg.cpu(), wu.cpu(), wd.cpu()
        per = time_oracle(xs_h, deps_h, wr_h, wg_h, wu_h, wd_h, shape, routing, args.cpu_trees)
        procs = max(1, host_cores())
        pool = OraclePool(procs, xs_h.clone(), deps_h.clone(), wr_h, wg_h, wu_h, wd_h, shape,
                          routing)
        n_all = 2 * procs
        wall, _ = pool.run(procs, n_all)
        pool.close()
        cpu = {"value": round(n_all / wall, 4), "unit": UNIT, "cores": procs, "kind": "oracle",
               "sample": f"{n_all} whole trees of this workload (65 rows each), one per task "
                         f"over {procs} oracle processes on {cpu_model()}",
               "seconds": round(wall, 2),
               "single_core": {"value": round(len(per) / sum(per), 4), "cores": 1,
                               "sample": f"{len(per)} whole trees, one after another",
                               "seconds": round(sum(per), 2)}}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": round(sec / K * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded EAGLE-3-shaped trees, N(0,0.02) weights)",
        "config": dict(workload_config(shape, routing, wr_std), parallelism=f"replicas{world}",
                       launch="eager" if args.no_graph else
                       "CUDA graphs of the timed steps (captured after the eager warm-up)"),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": peak_kind,
                     "kernel": "expert stage: selection launch (with its L2 prefetch of the "
                               "root's experts), token gather, grouped SwiGLU experts",
                     "window": "CUDA events before the selection launch and after the "
                               "grouped-expert kernel, every step of a separate pass over the "
                               "same trees",
                     "algo_bytes_per_launch_mean": int(stage_bytes.mean()),
                     "stage_ms_mean": round(float(stage_ms.mean()), 5),
                     "timed_steps": K_ev,
                     "expert_kernel_only": {
                         "achieved": round(ffn_only, 1), "frac": round(ffn_only / peak, 4),
                         "ms_mean": round(float(ffn_ms.mean()), 5),
                         "note": "gather + expert kernel alone; gross: the same bytes, part "
                                 "of which the selection launch already brought into L2"},
                     "whole_step": {"bytes_per_step": int(step_bytes.mean()),
                                    "achieved": round(whole, 1),
                                    "frac": round(whole / peak, 4)},
                     "traffic_note": "ncu DRAM read+write of the grouped-expert kernel per "
                                     "launch, scaled to this run's mean union",
                     "kernel_source_sha": kernel_sha()},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches_per_step * K),
        "clocks": clocks,
        "union": {"mean": float(union.mean()), "min": int(union.min()), "max": int(union.max()),
                  "first_steps": union[:20].tolist(),
                  "natural_mean": float(inf[:, 0].mean()), "selected_mean": float(inf[:, 1].mean()),
                  "m_mean": float(inf[:, 2].mean()),
                  "reuse_mean": round(float(1 - union.mean() / assignments), 4),
                  "fp64_pass_trees": int(inf[:, 4].sum()),
                  f"{other}_union_mean": float(u_o.mean()),
                  f"{other}_value": round(whole_job_rate(Kv, world, sec_o), 2)},
        "router_std_0.1": peaked,
        "two_blocks_in_flight": pair,
    }
    print(json.dumps(line))


def ffn_launches(M, L, path):
    """Kernel launches of the grouped-expert stage per step: two on either path (CUDA
    cores: gate/up, then down; tensor cores: the token-row gather, then one persistent
    launch for gate/up and down)."""
    return 2


# ------------------------------------------------------------ reference arm

def run_reference(args):
    """The oracle as the reference arm: every step one whole tree of the headline workload
    (router, selection, permute, every expert assignment, combine), the trees spread over
    the host's cores as independent processes. value = K / wall time of the K timed
    trees (the W warm-up trees run first, untimed)."""
    from expert_select_gb300 import workload as W
    from oracle import oracle as O

    world, rank, _ = dist_env()
    if rank != 0:
        return
    O.build()
    shape = W.QWEN3_30B_A3B
    xs_h, deps_h = make_trees(TREES, shape, SEED)
    wr = W.router_weight(SEED + 1, shape, std=args.router_std)
    wg, wu, wd = W.expert_weights(SEED + 2, shape)
    # a tree takes ~1.3 s on one core: beyond REF_MAX_TREES timed trees (about a minute
    # on 16 cores) the rate is taken on the first REF_MAX_TREES of the requested steps
    steps = min(args.steps, REF_MAX_TREES)
    warm = min(args.warmup, REF_MAX_WARMUP)
    procs = max(1, min(host_cores(), steps))
    pool = OraclePool(procs, xs_h, deps_h, wr, wg, wu, wd, shape, args.routing)
    pool.run(0, warm)
    wall, per = pool.run(warm, steps)
    pool.close()
    value = steps / wall
    sample = (f"per step: one whole tree of this workload (65 rows: router, selection, all "
              f"{65 * shape.k} expert assignments, combine); {steps} trees timed"
              f"{'' if steps == args.steps else f' of the {args.steps} requested'} over "
              f"{procs} oracle processes on {cpu_model()}, after {warm} warm-up trees; "
              f"mean {np.mean(per):.3f} s per tree per core")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": steps, "warmup": warm,
        "ms_per_step": round(wall / steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded EAGLE-3-shaped trees, N(0,0.02) weights)",
        "config": dict(workload_config(shape, args.routing, args.router_std),
                       parallelism=f"replicas{world}"),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": procs,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


# ------------------------------------------------------- secondary workloads
# Each prints one JSON line with the same contract keys as the headline line.

def _setup_gpu():
    import torch
    from expert_select_gb300 import build
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    return world, rank, local, torch.device("cuda", local)


def _timed(fn, dev, world):
    """Runs fn() between synchronised CUDA events; max over ranks (seconds)."""
    import torch
    s = torch.cuda.current_stream(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    fn()
    b.record(s)
    torch.cuda.synchronize(dev)
    barrier(world)
    return max_over_ranks(a.elapsed_time(b) / 1e3, world)


def _line(metric, value, unit, world, K, Wm, sec, config, **extra):
    d = {"metric": metric, "value": round(value, 3), "unit": unit, "n_gpus": world, "steps": K,
         "warmup": Wm, "ms_per_step": round(sec / K * 1e3, 4), "higher_is_better": True,
         "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
         "data": "synthetic (seeded EAGLE-3-shaped trees, N(0,0.02) weights)", "config": config}
    d.update(extra)
    return json.dumps(d)


def run_stack48(args):
    """48 independent Qwen3-shaped layers resident in HBM (~58 GB of experts), one fresh
    65-node tree per step through all layers with a pre-norm residual chain
    x <- x + MoE_l(rmsnorm(x)), as the target model's blocks are built (without the norm
    the residual stream of random layers grows until bf16 overflows)."""
    import torch
    from expert_select_gb300 import moetree as M
    from expert_select_gb300 import workload as W
    world, rank, local, dev = _setup_gpu()
    shape = W.QWEN3_30B_A3B
    NL = args.layers or 48
    seed = SEED + 2000 + 7919 * rank
    xs_h, deps_h = make_trees(TREES, shape, seed)
    xs, deps = xs_h.to(dev), deps_h.to(dev).int()
    layers = []
    for l in range(NL):
        wr = W.router_weight(seed + 10 ** 6 * (l + 1), shape, std=args.router_std, device=dev)
        wg, wu, wd = W.expert_weights(seed + 10 ** 6 * (l + 1) + 1, shape, device=dev)
        layers.append((wr, wg, wu, wd))
    N = xs.shape[1]
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    mode = M.MOE_ROUTE_ACCEPT if args.routing == "acceptmoe" else M.MOE_ROUTE_NATURAL
    P = M.select_params(mode, W.C_EAGLE)
    ws = M.workspace(L, 1, N, device=dev)
    x = torch.empty_like(xs[0])
    K, Wm = args.steps, args.warmup
    counts = torch.zeros(K, NL, shape.E, dtype=torch.int32, device=dev)
    info = torch.zeros(K, NL, M.MOE_INFO_FIELDS, dtype=torch.int32, device=dev)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(NL)] for _ in range(K)]
    s = torch.cuda.current_stream(dev)
    for row in ev:
        for a, b in row:
            a.record(s)
            b.record(s)
    torch.cuda.synchronize(dev)

    def step(i, record):
        x.copy_(xs[i % TREES])
        for l, (wr, wg, wu, wd) in enumerate(layers):
            out = M.tree_outputs(counts=counts[i, l], info=info[i, l]) if record else None
            opts = M.run_opts(args.ffn_path, ev[i][l][0], ev[i][l][1], residual=True,
                              norm_input=True) if record \
                else M.run_opts(args.ffn_path, residual=True, norm_input=True)
            M.moe_tree_forward(L, P, x, wr, wg, wu, wd, None, deps[i % TREES], 1, N, None, x,
                               ws, out, opts)

    for i in range(Wm):
        step(i, False)
    # the timed pass runs the layers alone; a second pass over the same trees records the
    # counters and the events around every expert kernel (an event between two launches
    # keeps the second from starting early, so it must not sit in the timed pass)
    with ClockSampler(local) as clk:
        sec = _timed(lambda: [step(i, False) for i in range(K)], dev, world)
    for i in range(K):
        step(i, True)
    torch.cuda.synchronize(dev)
    ffn_s = sum(a.elapsed_time(b) for row in ev for a, b in row) / 1e3
    union = (counts.cpu().numpy() > 0).sum(axis=2)  # [K, NL]

    # two trees in flight (two requests): even trees on this stream, odd ones on a second,
    # each with its own hidden state and workspace, the expert kernel capped to leave
    # --pair-free-sms SMs to the other tree's routing kernels
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    cap = max(1, nsm - args.pair_free_sms)
    s2 = torch.cuda.Stream(dev)
    x2 = torch.empty_like(x)
    ws2 = M.workspace(L, 1, N, device=dev)
    popts = M.run_opts(args.ffn_path, residual=True, norm_input=True, ffn_max_ctas=cap)

    def pair_steps(n):
        s2.wait_stream(s)
        for i in range(n):
            st, xb, wsb = (s, x, ws) if i % 2 == 0 else (s2, x2, ws2)
            with torch.cuda.stream(st):
                xb.copy_(xs[i % TREES])
            for wr, wg, wu, wd in layers:
                M.moe_tree_forward(L, P, xb, wr, wg, wu, wd, None, deps[i % TREES], 1, N, None,
                                   xb, wsb, None, popts, st)
        s.wait_stream(s2)

    pair_steps(Wm)
    torch.cuda.synchronize(dev)
    sec_pair = _timed(lambda: pair_steps(K), dev, world)
    algo = float((union * shape.expert_bytes).sum() + K * NL * 2 * N * shape.d * 2)
    peak, kind = measured_peaks()
    if rank == 0:
        print(_line("MoE verify, 48-layer stack: tree-blocks/s through all layers",
                    whole_job_rate(K, world, sec), "tree-blocks/s", world, K, Wm, sec,
                    {"workload": f"qwen3-30b-a3b-{NL}-layer-stack-resident", "layers": NL,
                     "routing": args.routing, "router_std": args.router_std,
                     "block": "x + MoE(rmsnorm(x))",
                     "expert_bytes_resident_gb": round(NL * shape.E * shape.expert_bytes / 1e9, 1),
                     "l2": "inputs larger than L2 (0.7 GB of union weights per layer)"},
                    per_layer_blocks_per_s=round(whole_job_rate(K, world, sec) * NL, 1),
                    two_blocks_in_flight={"value": round(whole_job_rate(K, world, sec_pair), 3),
                                          "streams": 2, "ffn_ctas": cap},
                    roofline={"bound": "hbm", "achieved": round(algo / ffn_s / 1e9, 1),
                              "peak": peak, "unit": "GB/s",
                              "frac": round(algo / ffn_s / 1e9 / peak, 4), "peak_kind": kind,
                              "kernel": "grouped SwiGLU experts"},
                    union={"mean": float(union.mean()), "min": int(union.min()),
                           "max": int(union.max())},
                    fp64_pass_frac=round(float(info[:, :, 4].float().mean().item()), 4),
                    clocks=clk.summary()))


def _pinned_empty(shape, dtype):
    """A host tensor of exactly this size, page-locked in place (cudaHostRegister)."""
    import torch
    t = torch.empty(shape, dtype=dtype)
    rc = torch.cuda.cudart().cudaHostRegister(t.data_ptr(), t.numel() * t.element_size(), 0)
    if int(rc) != 0:
        raise RuntimeError(f"cudaHostRegister failed ({rc})")
    return t


def run_offload(args):
    """GPT-OSS-120B-shaped layers with experts offloaded: `slots` expert slots per layer
    on the GPU, every expert in pinned host memory, uploads on a side stream. Per routing
    mode: H2D bytes, hit rate, and the share of the step the compute stream spent waiting
    for uploads ("AcceptMoE" news article, section 03: 65-78% under Standard SD, 27-35%
    with AcceptMoE, on an RTX 5090 over PCIe). Each step ends with a host read of that
    step's wait events. The three modes run interleaved, step by step (each with its own
    residency table and slot pools, in rotating order), so that the host link of a shared
    machine, whose rate drifts over minutes, affects them alike."""
    import torch
    from expert_select_gb300 import moetree as M
    from expert_select_gb300 import workload as W
    world, rank, local, dev = _setup_gpu()
    shape = W.GPT_OSS_120B
    NL = args.layers or 8
    slots = args.slots
    seed = SEED + 3000 + 7919 * rank
    xs_h, deps_h = make_trees(TREES, shape, seed)
    xs, deps = xs_h.to(dev), deps_h.to(dev).int()
    modes = (("natural", M.MOE_ROUTE_NATURAL, False),
             ("acceptmoe", M.MOE_ROUTE_ACCEPT, False),
             ("acceptmoe+prune", M.MOE_ROUTE_ACCEPT, True))
    t0 = time.perf_counter()
    layers = []
    for l in range(NL):
        wr = W.router_weight(seed + 10 ** 6 * (l + 1), shape, std=args.router_std, device=dev)
        wg, wu, wd = W.expert_weights(seed + 10 ** 6 * (l + 1) + 1, shape, device=dev)
        host = [_pinned_empty(w.shape, w.dtype) for w in (wg, wu, wd)]
        for h, w in zip(host, (wg, wu, wd)):
            h.copy_(w)
        del wg, wu, wd
        pools = [[torch.empty(slots, shape.f, shape.d, dtype=torch.bfloat16, device=dev),
                  torch.empty(slots, shape.f, shape.d, dtype=torch.bfloat16, device=dev),
                  torch.empty(slots, shape.d, shape.f, dtype=torch.bfloat16, device=dev)]
                 for _ in modes]
        layers.append((wr, host, pools))
    torch.cuda.empty_cache()
    setup_s = time.perf_counter() - t0
    # host link bandwidth: one 1 GiB pinned -> device copy
    hb = layers[0][1][0].view(-1)[: 1 << 29]
    db = torch.empty_like(hb, device=dev)
    db.copy_(hb)
    torch.cuda.synchronize(dev)
    link_s = _timed(lambda: db.copy_(hb, non_blocking=True), dev, 1)
    link_gbs = hb.numel() * 2 / link_s / 1e9
    del db
    N = xs.shape[1]
    Ls = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16", slots=slots)
    ws = M.workspace(Ls, 1, N, device=dev)
    x = torch.empty_like(xs[0])
    side = torch.cuda.Stream(dev)
    K, Wm = args.steps, args.warmup
    opts = M.run_opts(residual=True, norm_input=True)
    state = []
    for name, mode, prune in modes:
        P = M.select_params(mode, W.C_EAGLE, prune=prune, reroute_budget=8, min_set=16)
        state.append({"name": name, "P": P, "stats": [], "waits": [], "sec": 0.0,
                      "table": M.Residency(n_layers=NL, E=shape.E, slots=slots)})

    def step(m, i, keep):
        st_ = state[m]
        x.copy_(xs[i % TREES])
        for l, (wr, host, pools) in enumerate(layers):
            st = M.moe_offload_forward(Ls, st_["P"], x, wr, *host, *pools[m], st_["table"], l,
                                       deps[i % TREES], 1, N, x, ws, opts=opts,
                                       side_stream=side)
            if keep:
                st_["stats"].append((st.needed, st.hits, st.uploads, st.h2d_bytes, st.passes))
        if keep:  # the compute stream's upload waits of this step, layer by layer
            st_["waits"].append(sum(st_["table"].upload_wait(l)[0] for l in range(NL)))

    for i in range(Wm):
        for m in range(len(modes)):
            step(m, i, False)
    for i in range(K):
        for j in range(len(modes)):
            m = (i + j) % len(modes)
            state[m]["sec"] += _timed(lambda: step(m, i, True), dev, world)
    results = {}
    for st_ in state:
        a = np.array(st_["stats"], dtype=np.float64)
        sec, waits = st_["sec"], st_["waits"]
        h2d = float(a[:, 3].sum()) / K
        results[st_["name"]] = {
            "tree_blocks_per_s": round(K / sec, 3),
            "ms_per_step": round(sec / K * 1e3, 3),
            "needed_per_layer": round(float(a[:, 0].mean()), 2),
            "hit_rate": round(float(a[:, 1].sum() / a[:, 0].sum()), 4),
            "uploads_per_layer": round(float(a[:, 2].mean()), 2),
            "h2d_gb_per_step": round(h2d / 1e9, 3),
            "passes_per_layer": round(float(a[:, 4].mean()), 2),
            "upload_wait_ms_per_step": round(float(np.mean(waits)), 3),
            "upload_wait_frac": round(float(np.sum(waits) / 1e3 / sec), 4),
            "upload_gbs_while_waiting": round(h2d / max(float(np.mean(waits)) / 1e3, 1e-9) / 1e9, 1)}
        st_["table"].close()
    nat = results["natural"]
    for name in ("acceptmoe", "acceptmoe+prune"):
        r = results[name]
        r["speedup_vs_natural"] = round(r["tree_blocks_per_s"] / nat["tree_blocks_per_s"], 3)
        r["h2d_reduction_vs_natural"] = round(
            1 - r["h2d_gb_per_step"] / max(nat["h2d_gb_per_step"], 1e-12), 4)
        r["hit_rate_gain_pp"] = round(100 * (r["hit_rate"] - nat["hit_rate"]), 2)
    main_r = results["acceptmoe+prune"]
    if rank == 0:
        print(_line("MoE verify with expert offload: tree-blocks/s through all layers",
                    main_r["tree_blocks_per_s"] * world, "tree-blocks/s", world, K, Wm,
                    K / main_r["tree_blocks_per_s"],
                    {"workload": f"gpt-oss-120b-{NL}-layer-offload-{slots}-slots",
                     "layers": NL, "slots": slots, "router_std": args.router_std,
                     "block": "x + MoE(rmsnorm(x))",
                     "routing": "acceptmoe + residency-aware pruning (budget 8, min 16)",
                     "modes_interleaved": True,
                     "host_store_gb": round(NL * shape.E * shape.expert_bytes / 1e9, 1)},
                    modes=results, h2d_link_gbs=round(link_gbs, 1), setup_s=round(setup_s, 1)))


def run_batched(args):
    """The Qwen3-shaped layer with B independent 65-node trees per verification block."""
    import torch
    from expert_select_gb300 import moetree as M
    from expert_select_gb300 import workload as W
    world, rank, local, dev = _setup_gpu()
    shape = W.QWEN3_30B_A3B
    seed = SEED + 4000 + 7919 * rank
    Bs = [int(b) for b in args.batches.split(",")]
    n_trees = max(TREES, 2 * max(Bs))
    xs_h, deps_h = make_trees(n_trees, shape, seed)
    xs, deps = xs_h.to(dev), deps_h.to(dev).int()
    wr = W.router_weight(seed + 1, shape, std=args.router_std, device=dev)
    wg, wu, wd = W.expert_weights(seed + 2, shape, device=dev)
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    N = xs.shape[1]
    peak, kind = measured_peaks()
    tflops_peak = 1934.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            tflops_peak = float(json.load(fh)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        pass
    rows = []
    K, Wm = args.steps, args.warmup
    for B in Bs:
        R = B * N
        ws = M.workspace(L, B, N, device=dev)
        y = torch.empty(R, shape.d, dtype=torch.bfloat16, device=dev)
        nblk = n_trees // B
        xb = [xs[j * B:(j + 1) * B].reshape(R, shape.d) for j in range(nblk)]
        db = [deps[j * B:(j + 1) * B].reshape(R) for j in range(nblk)]
        for routing, mode in (("natural", M.MOE_ROUTE_NATURAL), ("acceptmoe", M.MOE_ROUTE_ACCEPT)):
            P = M.select_params(mode, W.C_EAGLE)
            counts = torch.zeros(K, shape.E, dtype=torch.int32, device=dev)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
            s = torch.cuda.current_stream(dev)
            for a, b in ev:
                a.record(s)
                b.record(s)

            def loop(n, rec):
                for i in range(n):
                    j = i % nblk
                    M.moe_tree_forward(L, P, xb[j], wr, wg, wu, wd, None, db[j], B, N, None, y,
                                       ws, M.tree_outputs(counts=counts[i]) if rec else None,
                                       M.run_opts(args.ffn_path, ev[i][0], ev[i][1]) if rec
                                       else None)

            loop(Wm, False)
            sec = _timed(lambda: loop(K, True), dev, world)
            ffn_s = sum(a.elapsed_time(b) for a, b in ev) / 1e3
            c = counts.cpu().numpy()
            union = (c > 0).sum(axis=1)
            A = c.sum(axis=1)
            algo = float((union * shape.expert_bytes).sum() + K * 2 * R * shape.d * 2)
            flops = float((2.0 * A * 3 * shape.d * shape.f).sum())
            rows.append({"B": B, "rows": R, "routing": routing,
                         "blocks_per_s": round(whole_job_rate(K, world, sec), 2),
                         "trees_per_s": round(whole_job_rate(K, world, sec) * B, 1),
                         "ms_per_block": round(sec / K * 1e3, 4),
                         "ffn_ms": round(ffn_s / K * 1e3, 4), "union": round(float(union.mean()), 2),
                         "tokens_per_expert": round(float((A / np.maximum(union, 1)).mean()), 1),
                         "ffn_gbs": round(algo / ffn_s / 1e9, 1),
                         "ffn_hbm_frac": round(algo / ffn_s / 1e9 / peak, 4),
                         "ffn_tflops": round(flops / ffn_s / 1e12, 1),
                         "ffn_tensor_frac": round(flops / ffn_s / 1e12 / tflops_peak, 4)})
    if rank == 0:
        best = rows[-1]
        print(_line("MoE verify layer, batched trees: tree-blocks/s", best["blocks_per_s"],
                    "tree-blocks/s", world, K, Wm, 1.0 / best["blocks_per_s"] * K,
                    {"workload": "qwen3-30b-a3b-moe-layer-batched-trees", "batches": Bs,
                     "router_std": args.router_std,
                     "l2": "inputs larger than L2 (>= 0.7 GB of union weights per block)"},
                    sweep=rows, hbm_peak=peak, bf16_tflops_peak=tflops_peak))


def _layer_setup(args, seed_off):
    import torch
    from expert_select_gb300 import moetree as M
    from expert_select_gb300 import workload as W
    world, rank, local, dev = _setup_gpu()
    shape = W.QWEN3_30B_A3B
    seed = SEED + seed_off + 7919 * rank
    xs_h, deps_h = make_trees(TREES, shape, seed)
    xs, deps = xs_h.to(dev), deps_h.to(dev).int()
    wr = W.router_weight(seed + 1, shape, std=args.router_std, device=dev)
    wg, wu, wd = W.expert_weights(seed + 2, shape, device=dev)
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    return torch, M, W, world, rank, local, dev, shape, xs, deps, wr, wg, wu, wd, L


def run_budget(args):
    """Fixed-budget selection rules beside AcceptMoE on the Qwen3-shaped layer ("AcceptMoE"
    news article, section 04): AcceptMoE-B (commitment-weighted demand, set size B) and the
    MoE-Spec rule (uniform position weights, no anchor, set size B). Only the cost side is
    measurable without trained models: union size and verify throughput."""
    (torch, M, W, world, rank, local, dev, shape, xs, deps, wr, wg, wu, wd, L) = \
        _layer_setup(args, 5000)
    N = xs.shape[1]
    ws = M.workspace(L, 1, N, device=dev)
    y = torch.empty(N, shape.d, dtype=torch.bfloat16, device=dev)
    K, Wm = args.steps, args.warmup
    variants = [("natural", M.select_params(M.MOE_ROUTE_NATURAL, W.C_EAGLE)),
                ("acceptmoe", M.select_params(M.MOE_ROUTE_ACCEPT, W.C_EAGLE))]
    for B in (16, 24, 32):
        variants.append((f"acceptmoe-B{B}", M.select_params(M.MOE_ROUTE_FIXED_B, W.C_EAGLE,
                                                           fixed_B=B)))
        variants.append((f"moe-spec-B{B}", M.select_params(M.MOE_ROUTE_FIXED_B, [1.0],
                                                           anchor=False, fixed_B=B)))
    rows = []
    for name, P in variants:
        info = torch.zeros(K, M.MOE_INFO_FIELDS, dtype=torch.int32, device=dev)

        def loop(n, rec):
            for i in range(n):
                j = i % TREES
                M.moe_tree_forward(L, P, xs[j], wr, wg, wu, wd, None, deps[j], 1, N, None, y,
                                   ws, M.tree_outputs(info=info[i]) if rec else None)

        loop(Wm, False)
        sec = _timed(lambda: loop(K, True), dev, world)
        inf = info.cpu().numpy()
        rows.append({"rule": name, "blocks_per_s": round(whole_job_rate(K, world, sec), 1),
                     "union": round(float(inf[:, 1].mean()), 2),
                     "set_size": round(float(inf[:, 2].mean()), 2)})
    if rank == 0:
        acc = next(r for r in rows if r["rule"] == "acceptmoe")
        print(_line("MoE verify layer tree-blocks/s under fixed-budget selection rules",
                    acc["blocks_per_s"], "tree-blocks/s", world, K, Wm,
                    K / acc["blocks_per_s"],
                    {"workload": "qwen3-30b-a3b-moe-layer-resident-eagle3-tree",
                     "router_std": args.router_std},
                    rules=rows))


def run_efficiency(args):
    """Target efficiency eta(N) = T(1 row) / T(N rows) of the layer (MoESD notes, section
    5.2), the N rows being the first N nodes of each tree (parents come first, so every
    prefix is itself a tree), natural routing as in plain verification."""
    (torch, M, W, world, rank, local, dev, shape, xs, deps, wr, wg, wu, wd, L) = \
        _layer_setup(args, 6000)
    K, Wm = args.steps, args.warmup
    P = M.select_params(M.MOE_ROUTE_NATURAL, W.C_EAGLE)
    rows = []
    for n in (1, 2, 4, 8, 16, 33, 65):
        ws = M.workspace(L, 1, n, device=dev)
        y = torch.empty(n, shape.d, dtype=torch.bfloat16, device=dev)
        xb = [xs[j, :n].contiguous() for j in range(TREES)]
        db = [deps[j, :n].contiguous() for j in range(TREES)]
        counts = torch.zeros(K, shape.E, dtype=torch.int32, device=dev)

        def loop(m, rec):
            for i in range(m):
                j = i % TREES
                M.moe_tree_forward(L, P, xb[j], wr, wg, wu, wd, None, db[j], 1, n, None, y, ws,
                                   M.tree_outputs(counts=counts[i]) if rec else None)

        loop(Wm, False)
        sec = _timed(lambda: loop(K, True), dev, world)
        union = (counts.cpu().numpy() > 0).sum(axis=1)
        rows.append({"rows": n, "ms_per_block": round(sec / K * 1e3, 4),
                     "union": round(float(union.mean()), 2)})
    t1 = rows[0]["ms_per_block"]
    for r in rows:
        r["eta"] = round(t1 / r["ms_per_block"], 4)
        r["expected_union_uniform"] = round(shape.E * (1 - ((shape.E - shape.k) / shape.E)
                                                       ** r["rows"]), 2)
    if rank == 0:
        print(_line("MoE verify layer target efficiency T(1 row)/T(N rows)", rows[-1]["eta"],
                    "ratio", world, K, Wm, rows[-1]["ms_per_block"] * K / 1e3,
                    {"workload": "qwen3-30b-a3b-moe-layer-tree-prefixes",
                     "router_std": args.router_std}, sweep=rows))


def run_ecospec(args):
    """Cost-aware choice of the verified tree (EcoSpec stand-in) on the Qwen3-shaped layer:
    per step, the router over all ~411 drafted candidates gives each candidate's predicted
    footprint (its natural top-k), moe_draft_select picks 65 nodes with
    log P - lambda * (new experts), and the chosen tree is verified with natural routing.
    lambda = 0 is the confidence-ordered tree (the EAGLE-3 stand-in)."""
    import torch
    from expert_select_gb300 import moetree as M
    from expert_select_gb300 import workload as W
    world, rank, local, dev = _setup_gpu()
    shape = W.QWEN3_30B_A3B
    seed = SEED + 7000 + 7919 * rank
    n_pools = 16
    pools = []
    for i in range(n_pools):
        c = W.eagle_candidates(seed + i)
        x = W.hidden_states(seed + 100 + i, c.parent, shape.d, torch.bfloat16).to(dev)
        td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        pools.append((c.C, td(c.parent), td(c.depth), td(c.logp), x))
    wr = W.router_weight(seed + 1, shape, std=args.router_std, device=dev)
    wg, wu, wd = W.expert_weights(seed + 2, shape, device=dev)
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    gamma = 65
    Cmax = max(p[0] for p in pools)
    logits = torch.empty(Cmax, shape.E, device=dev)
    fp = torch.empty(Cmax, shape.k, dtype=torch.int32, device=dev)
    g = torch.empty(Cmax, shape.k, device=dev)
    sel = torch.empty(gamma, dtype=torch.int32, device=dev)
    spar, sdep = torch.empty_like(sel), torch.empty_like(sel)
    x_sel = torch.empty(gamma, shape.d, dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(x_sel)
    ws = M.workspace(L, 1, gamma, device=dev)
    PN = M.select_params(M.MOE_ROUTE_NATURAL, [1.0])
    K, Wm = args.steps, args.warmup
    rows = []
    for lam in (0.0, 0.1, 0.3, 1.0):
        nu = torch.zeros(K, dtype=torch.int32, device=dev)
        cnt = torch.zeros(K, shape.E, dtype=torch.int32, device=dev)
        sel_k = torch.zeros(K, gamma, dtype=torch.int32, device=dev)
        cnt_v = torch.zeros(shape.E, dtype=torch.int32, device=dev)  # verify-only rounds

        def step(i, verify_only=False):
            C, par, dep, lp, x = pools[i % n_pools]
            if not verify_only:
                M.moe_router_logits(L, x, wr, logits[:C])
                M.moe_tree_select(L, PN, logits[:C], dep, 1, C, None, fp[:C], g[:C])
                M.moe_draft_select(L, par, dep, lp, fp[:C], lam, gamma, sel_k[i], spar, sdep,
                                   x, x_sel, nu[i])
            M.moe_tree_forward(L, PN, x_sel, wr, wg, wu, wd, None, sdep, 1, gamma, None, y, ws,
                               M.tree_outputs(counts=cnt_v if verify_only else cnt[i]))

        for i in range(Wm):
            step(i)
        sec = _timed(lambda: [step(i) for i in range(K)], dev, world)
        sec_v = _timed(lambda: [step(i, True) for i in range(K)], dev, world)
        mass = [float(pools[i % n_pools][3][sel_k[i].long()].sum()) for i in range(K)]
        union = (cnt.cpu().numpy() > 0).sum(axis=1)
        rows.append({"lambda": lam, "blocks_per_s": round(whole_job_rate(K, world, sec), 1),
                     "verify_only_blocks_per_s": round(whole_job_rate(K, world, sec_v), 1),
                     "verified_union": round(float(union.mean()), 2),
                     "predicted_union": round(float(nu.float().mean().item()), 2),
                     "sum_logp_selected": round(float(np.mean(mass)), 3)})
    if rank == 0:
        r0 = rows[0]
        for r in rows:
            r["union_vs_confidence"] = round(r["verified_union"] / r0["verified_union"], 4)
        print(_line("MoE verify with cost-aware draft selection: tree-blocks/s incl. selection",
                    rows[2]["blocks_per_s"], "tree-blocks/s", world, K, Wm,
                    K / rows[2]["blocks_per_s"],
                    {"workload": "qwen3-30b-a3b-layer-eagle3-candidates-ecospec",
                     "candidates": "all nodes of a 5-step top-10 expansion", "gamma": gamma,
                     "router_std": args.router_std}, sweep=rows))


def run_crossover(args):
    """The grouped-expert stage alone (moe_expert_forward) on the CUDA-core and tensor-core
    paths, with exactly r rows routed to each of 64 experts (r = 1 .. 256), Qwen3-shaped
    bf16 experts: where the batch regime turns from memory-bound to compute-bound (MoESD
    notes, section 5.1) and which path wins at each rows-per-expert count. Events bracket
    the expert launches of each call (CUDA cores: gate/up and down; tensor cores: the token
    gather and the expert kernel)."""
    import torch
    from expert_select_gb300 import moetree as M
    from expert_select_gb300 import workload as W
    world, rank, local, dev = _setup_gpu()
    shape = W.QWEN3_30B_A3B
    n_exp = 64
    wg, wu, wd = W.expert_weights(SEED + 8000, shape, device=dev)
    L = M.layer_desc(shape.d, shape.E, shape.k, shape.f, "bf16")
    peak, _ = measured_peaks()
    tflops_peak = 1895.9
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            tflops_peak = float(json.load(fh)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        pass
    K, Wm = args.steps, args.warmup
    s = torch.cuda.current_stream(dev)
    rows = []
    for r in (1, 2, 4, 8, 16, 32, 64, 128, 256):
        R = n_exp * r // shape.k
        t = torch.arange(R, device=dev).view(R, 1) * shape.k + torch.arange(shape.k, device=dev)
        idx = (t % n_exp).int().contiguous()  # every expert gets exactly r rows
        gates = torch.full((R, shape.k), 1.0 / shape.k, device=dev)
        x = W.hidden_states(SEED + 8001 + r, np.arange(-1, R - 1, dtype=np.int32), shape.d,
                            torch.bfloat16).to(dev)
        y = torch.empty_like(x)
        ws = M.workspace(L, 1, R, device=dev)
        A = R * shape.k
        bytes_ = n_exp * shape.expert_bytes + 2 * R * shape.d * 2
        flops = 2.0 * A * 3 * shape.d * shape.f
        res = {"rows_per_expert": r, "rows": R}
        for name, path in (("cuda_cores", M.MOE_FFN_SIMT), ("tcgen05", M.MOE_FFN_TCGEN05)):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
            for a, b in ev:
                a.record(s)
                b.record(s)
            for _ in range(Wm):
                M.moe_expert_forward(L, x, wg, wu, wd, None, idx, gates, y, ws, M.run_opts(path))
            torch.cuda.synchronize(dev)
            for i in range(K):
                M.moe_expert_forward(L, x, wg, wu, wd, None, idx, gates, y, ws,
                                     M.run_opts(path, ev[i][0], ev[i][1]))
            torch.cuda.synchronize(dev)
            ms = float(np.median([a.elapsed_time(b) for a, b in ev]))
            res[name] = {"ms": round(ms, 4),
                         "gbs": round(bytes_ / ms / 1e6, 1),
                         "hbm_frac": round(bytes_ / ms / 1e6 / peak, 4),
                         "tflops": round(flops / ms / 1e9, 1),
                         "tensor_frac": round(flops / ms / 1e9 / tflops_peak, 4)}
        res["faster"] = "tcgen05" if res["tcgen05"]["ms"] < res["cuda_cores"]["ms"] else \
            "cuda_cores"
        rows.append(res)
    if rank == 0:
        print(_line("grouped SwiGLU expert stage: CUDA cores vs tcgen05 by rows per expert",
                    rows[-1]["tcgen05"]["tflops"], "TFLOP/s", world, K, Wm,
                    rows[-1]["tcgen05"]["ms"] * K / 1e3,
                    {"workload": "qwen3-30b-a3b-experts-64-active-rows-per-expert-sweep",
                     "experts": n_exp, "l2": "604 MB of expert weights per call (> L2)"},
                    sweep=rows, hbm_peak=peak, bf16_tflops_peak=tflops_peak))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 5000; 200 for stack48 and offload, the "
                         "verification steps those workloads are defined over)")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--routing", choices=["acceptmoe", "natural"], default="acceptmoe")
    ap.add_argument("--router-std", type=float, default=0.02)
    ap.add_argument("--ffn-path", type=int, default=0, help="0 auto, 1 simt, 2 tcgen05")
    ap.add_argument("--cpu-trees", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the timed steps eagerly instead of from CUDA graphs")
    ap.add_argument("--workload", choices=["layer", "stack48", "offload", "batched", "budget",
                                           "efficiency", "ecospec", "crossover"],
                    default="layer", help="layer: the Qwen3-shaped layer (default line)")
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--slots", type=int, default=48)
    ap.add_argument("--batches", default="1,4,16,64")
    ap.add_argument("--pair-free-sms", type=int, default=8,
                    help="SMs the expert kernel leaves free when two blocks are in flight")
    args = ap.parse_args(argv)
    if args.steps is None:
        args.steps = 200 if args.workload in ("stack48", "offload") else 5000
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "stack48":
        run_stack48(args)
    elif args.workload == "offload":
        run_offload(args)
    elif args.workload == "batched":
        run_batched(args)
    elif args.workload == "budget":
        run_budget(args)
    elif args.workload == "efficiency":
        run_efficiency(args)
    elif args.workload == "ecospec":
        run_ecospec(args)
    elif args.workload == "crossover":
        run_crossover(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
