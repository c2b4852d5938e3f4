#!/usr/bin/env python
"""Throughput of the multi-LoRA delta path on one GB300 (or N, weak scaling).

One step = one pass of the whole path over one batch of synthetic input:
``lora_prepare_batch`` (device-side grouping) + ``lora_delta`` (fused shrink,
scale and expand), both through the C ABI.  Default workload: the decode
SGMV batch (256 single-token rows, 4096 -> 4096, rank 16, 32 of 64 pool
adapters active, bf16).

Timing: W eager warm-up steps, then exactly K steps captured in CUDA graphs
and replayed between CUDA events on the launching stream, bracketed by a
barrier and a device synchronize.  Every step uses one of S rotating input
sets (x, y, pools, ids, workspace) whose total exceeds L2, so no step finds
its inputs in L2.  The kernels of a step are chained by programmatic
dependent launch.  Kernel durations (for the roofline) come from one more
replay of the same steps in which event nodes bracket every call; event
nodes cut the programmatic overlap, so that replay is kept out of the timed
region.  When one kernel takes every active row (the tensor-core kernel on
prefill, the CUDA-core kernel on decode) a further replay forces the path to
it, so the roofline divides by that kernel's own launch time; otherwise by
the time of the whole lora_delta call.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from segmented_gather_gemv_gb300 import workloads as wl  # noqa: E402

METRIC = ("LoRA-delta tokens/s and achieved HBM GB/s (% of ~8 TB/s) "
          "for decode SGMV and prefill")
L2_BYTES = 129 * 1024 * 1024
NOMINAL_HBM_GBS = 8000.0
WORKLOADS = {
    "decode": (lambda seed: wl.decode(seed=seed), 50000),
    "prefill": (lambda seed: wl.prefill(seed=seed), 4000),
    "prefill_chunk64": (lambda seed: wl.prefill(seed=seed, chunk_size=64), 4000),
    "mixed_rank_up": (lambda seed: wl.mixed_rank(seed=seed, proj="up"), 20000),
    "mixed_rank_down": (lambda seed: wl.mixed_rank(seed=seed, proj="down"), 20000),
    "mixed_serving": (lambda seed: wl.mixed_serving(seed=seed), 10000),
}
# Kernel sources whose counters a committed ncu summary refers to.
KERNEL_SOURCES = {
    "sgmv_cc_kernel": ["segmented_gather_gemv_gb300/csrc/sgmv_cc.cu",
                       "segmented_gather_gemv_gb300/csrc/common.cuh"],
    "sgmv_tc_kernel": ["segmented_gather_gemv_gb300/csrc/sgmv_tc.cu",
                       "segmented_gather_gemv_gb300/csrc/common.cuh"],
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 CUDA cores, 2 tensor cores")
    ap.add_argument("--graph-steps", type=int, default=512)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def algorithmic_bytes(w: wl.Workload) -> dict:
    """Unique bytes the delta must move: active x rows, the touched adapters'
    A and B at their true rank, and the read + write of active y rows."""
    es = 2 if w.dtype == "bf16" else 4
    act = (w.ids >= 0) & (w.ids < w.n_adapters)
    n_act = int(act.sum())
    touched = np.unique(w.ids[act])
    ranks = (np.full(w.n_adapters, w.r_max) if w.ranks is None else w.ranks)[touched]
    x = n_act * w.d_in * es
    a = int(ranks.sum()) * w.d_in * es
    b = int(ranks.sum()) * w.d_out * es
    y = 2 * n_act * w.d_out * es
    a_pad = len(touched) * w.r_max * w.d_in * es
    b_pad = len(touched) * w.r_max * w.d_out * es
    return {"x": x, "A": a, "B": b, "y_rw": y, "total": x + a + b + y,
            "total_padded_rank": x + a_pad + b_pad + y, "active_rows": n_act,
            "touched_adapters": int(len(touched))}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES.get(kernel, []):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("source_sha256_16") != source_hash(kernel):
        return None
    return int(e["dram_bytes_per_launch"])


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        if not shutil.which("nvidia-smi"):
            return
        self.proc = subprocess.Popen(
            ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
             "--format=csv,noheader,nounits", "-lms", "100"],
            stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU side

def cpu_baseline(w: wl.Workload, seconds: float) -> dict:
    """The oracle, as it stands, on the host: full batches (prepare + delta)
    repeated until `seconds` have passed; single-threaded."""
    import oracle
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.prepare_batch(w.ids, w.n_adapters, w.chunk_size)
        oracle.delta(w.x, w.ids, w.A, w.B, w.y, scale=w.scale,
                     adapter_scale=w.adapter_scale, ranks=w.ranks)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": reps * w.M / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": "%d full batches of %d rows (grouping + fp64 per-token delta), %.1f s"
                      % (reps, w.M, dt)}


def replica_seed(rank: int) -> int:
    """Seed of rank `rank`'s batch: every replica draws its own batch (weak scaling)."""
    return 42 + rank


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(world: int, steps: int, rows_per_step: int, elapsed_ms: float) -> float:
    """Tokens of all ranks' timed steps over the slowest rank's time."""
    return world * steps * rows_per_step / (elapsed_ms / 1e3)


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    factory, default_steps = WORKLOADS[args.workload]
    w = factory(42)
    import oracle
    oracle.build()
    K = args.steps if args.steps is not None else 20
    W = max(3, args.warmup)
    # Per step: a bounded sample of the batch's rows, sized so the whole run
    # takes about two minutes at most.
    t0 = time.perf_counter()
    oracle.delta(w.x[:8], w.ids[:8], w.A, w.B, w.y[:8], scale=w.scale,
                 adapter_scale=w.adapter_scale, ranks=w.ranks)
    per_row = max((time.perf_counter() - t0) / 8, 1e-6)
    rows = int(max(1, min(w.M, 100.0 / (K + W) / per_row)))
    sel = np.arange(rows)

    def step():
        oracle.prepare_batch(w.ids[sel], w.n_adapters, w.chunk_size)
        oracle.delta(w.x[sel], w.ids[sel], w.A, w.B, w.y[sel], scale=w.scale,
                     adapter_scale=w.adapter_scale, ranks=w.ranks)

    for _ in range(W):
        step()
    t0 = time.perf_counter()
    for _ in range(K):
        step()
    dt = time.perf_counter() - t0
    value = K * rows / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": 1e3 * dt / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "tokens_per_step": rows,
                   "sample": "first %d of %d rows per step" % (rows, w.M)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "first %d of %d rows of %s per step, %d steps"
                                   % (rows, w.M, w.name, K)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU side

def run_ours(args, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist
    from segmented_gather_gemv_gb300 import binding as B

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    factory, default_steps = WORKLOADS[args.workload]
    K = args.steps if args.steps is not None else default_steps
    W = max(3, args.warmup)
    w = factory(replica_seed(rank))
    es = 2 if w.dtype == "bf16" else 4
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    ab = algorithmic_bytes(w)

    # Rotating input sets: enough copies that the sets together exceed L2.
    set_bytes = (w.x.size + w.y.size + w.A.size + sum(b.size for b in w.B)) * es
    n_sets = int(min(64, max(2, math.ceil(3 * L2_BYTES / set_bytes))))
    x0 = torch.from_numpy(w.x).to(dev, tdt)
    y0 = torch.from_numpy(w.y).to(dev, tdt)
    A0 = torch.from_numpy(w.A).to(dev, tdt)
    B0 = [torch.from_numpy(b).to(dev, tdt) for b in w.B]
    ids0 = torch.from_numpy(w.ids).to(dev)
    ranks = None if w.ranks is None else torch.from_numpy(w.ranks).to(dev)
    ascale = None if w.adapter_scale is None else torch.from_numpy(w.adapter_scale).to(dev)
    ws_bytes = B.lora_workspace_size(w.M, w.n_adapters, w.chunk_size)
    sets = []
    for i in range(n_sets):
        sets.append({
            "x": x0 if i == 0 else x0.clone(), "y": y0 if i == 0 else y0.clone(),
            "A": A0 if i == 0 else A0.clone(), "B": B0 if i == 0 else [b.clone() for b in B0],
            "ids": ids0 if i == 0 else ids0.clone(),
            "ws": torch.empty(ws_bytes, dtype=torch.uint8, device=dev),
        })
    stream = torch.cuda.Stream(device=dev)

    def step(s):
        batch = B.lora_prepare_batch(s["ids"], w.n_adapters, w.chunk_size, workspace=s["ws"],
                                     stream=stream)
        B.lora_delta(batch, s["x"], s["A"], s["B"], s["y"], scale=w.scale,
                     adapter_scale=ascale, ranks=ranks, path=args.path, stream=stream)
        return batch

    with torch.cuda.stream(stream):
        for i in range(W):
            step(sets[i % n_sets])
    stream.synchronize()
    b0 = B.lora_prepare_batch(sets[0]["ids"], w.n_adapters, w.chunk_size, workspace=sets[0]["ws"],
                              stream=stream)
    stream.synchronize()
    counts = b0.counts()
    n_launch0 = B.lora_launch_count()
    step(sets[0])
    launches_per_step = B.lora_launch_count() - n_launch0
    stream.synchronize()

    # Graphs of G steps with event nodes around each kernel.
    G = max(1, min(args.graph_steps, K))
    use_graph = True
    try:
        probe = torch.cuda.Event(enable_timing=True, external=True)
        del probe
    except TypeError:
        use_graph = False

    # The dominant kernel alone: when one kernel takes every active row, the
    # path forced to it launches exactly that kernel with the same work.
    dom_path = None
    if args.path == 0 and counts["num_active"] > 0:
        if counts["tc_rows"] == counts["num_active"]:
            dom_path = 2
        elif counts["tc_rows"] == 0:
            dom_path = 1

    def capture(nsteps, offset, timed, path=None):
        """Graph of `nsteps` steps.  With `timed`, event nodes bracket every
        kernel (they also cut the programmatic overlap between kernels, so
        the step-time graph has none)."""
        path = args.path if path is None else path
        evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True)) for _ in range(nsteps if timed else 0)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(nsteps):
                s = sets[(offset + i) % n_sets]
                if timed:
                    evs[i][0].record(stream)
                batch = B.lora_prepare_batch(s["ids"], w.n_adapters, w.chunk_size,
                                             workspace=s["ws"], stream=stream)
                if timed:
                    evs[i][1].record(stream)
                B.lora_delta(batch, s["x"], s["A"], s["B"], s["y"], scale=w.scale,
                             adapter_scale=ascale, ranks=ranks, path=path, stream=stream)
                if timed:
                    evs[i][2].record(stream)
        return g, evs

    reps, rem = divmod(K, G)
    if use_graph:
        g_main, _ = capture(G, 0, False)
        g_rem, _ = capture(rem, 0, False) if rem else (None, [])
        g_kern, ev_main = capture(G, 0, True)
        g_dom, ev_dom = capture(G, 0, True, dom_path) if dom_path is not None else (None, [])
        with torch.cuda.stream(stream):
            g_main.replay()
            g_kern.replay()
            if g_dom is not None:
                g_dom.replay()
        stream.synchronize()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    clocks = ClockSampler(vis.split(",")[local_rank].strip() if vis else str(local_rank))
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    t_start.record(stream)
    if use_graph:
        with torch.cuda.stream(stream):     # a graph replays on the current stream
            for _ in range(reps):
                g_main.replay()
            if g_rem is not None:
                g_rem.replay()
    else:
        with torch.cuda.stream(stream):
            for i in range(K):
                step(sets[i % n_sets])
    t_end.record(stream)
    t_end.synchronize()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)

    # Kernel durations: the same steps replayed once more with event nodes
    # around every kernel, right after the timed region.
    prep_us, delta_us, dom_us = [], [], []
    if use_graph:
        with torch.cuda.stream(stream):
            g_kern.replay()
            if g_dom is not None:
                g_dom.replay()
        stream.synchronize()
        for e0, e1, e2 in ev_main:
            prep_us.append(1e3 * e0.elapsed_time(e1))
            delta_us.append(1e3 * e1.elapsed_time(e2))
        for e0, e1, e2 in ev_dom:
            dom_us.append(1e3 * e1.elapsed_time(e2))
    ms_per_step = elapsed_ms / K
    value = whole_job_tokens_per_s(world, K, w.M, elapsed_ms)

    # e2e: the public API from pinned host buffers, copies inside the region.
    x_h = torch.from_numpy(w.x).to(tdt).pin_memory()
    y_h = torch.from_numpy(w.y).to(tdt).pin_memory()
    ids_h = torch.from_numpy(w.ids).pin_memory()
    y_out = torch.empty_like(y_h).pin_memory()
    s0 = sets[0]
    E = args.e2e_steps
    with torch.cuda.stream(stream):
        for i in range(3 + E):
            if i == 3:
                stream.synchronize()
                e_a = torch.cuda.Event(enable_timing=True)
                e_b = torch.cuda.Event(enable_timing=True)
                e_a.record(stream)
            s0["x"].copy_(x_h, non_blocking=True)
            s0["y"].copy_(y_h, non_blocking=True)
            s0["ids"].copy_(ids_h, non_blocking=True)
            step(s0)
            y_out.copy_(s0["y"], non_blocking=True)
        e_b.record(stream)
    e_b.synchronize()
    e2e_ms = e_a.elapsed_time(e_b) / E
    h2d = (x_h.numel() + y_h.numel()) * es + ids_h.numel() * 4
    d2h = y_out.numel() * es

    peak, peak_kind = load_peaks()
    d_us = statistics.mean(delta_us) if delta_us else None
    k_us = statistics.mean(dom_us) if dom_us else d_us
    achieved = ab["total"] / (k_us * 1e-6) / 1e9 if k_us else None
    # dominant kernel: the tensor-core one when most active rows are in its segments
    kernel = "sgmv_tc_kernel" if 2 * counts["tc_rows"] > max(1, counts["num_active"]) else "sgmv_cc_kernel"
    traffic = committed_traffic(kernel, args.workload)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {
            "workload": w.name, "tokens_per_step": w.M, "active_rows": ab["active_rows"],
            "touched_adapters": ab["touched_adapters"], "num_segs": counts["num_segs"],
            "chunk_size": w.chunk_size, "path": ["auto", "cuda_core", "tensor"][args.path],
            "l2": "inputs rotate over %d sets (%.0f MB > %d MB L2)"
                  % (n_sets, n_sets * set_bytes / 1e6, L2_BYTES // 2**20),
            "timing": ("CUDA graphs of %d steps (kernels chained by programmatic dependent "
                       "launch); kernel durations from a replay of the same steps with event "
                       "nodes around each kernel" % G) if use_graph else "eager launches",
            "parallelism": "replicas: one independent batch per GPU" if world > 1 else "single GPU",
        },
        "kernels_us": {"prepare_mean": statistics.mean(prep_us) if prep_us else None,
                       "delta_mean": d_us,
                       "delta_median": statistics.median(delta_us) if delta_us else None,
                       "kernel_mean": k_us},
        "algorithmic_bytes_per_step": ab["total"],
        "algorithmic_bytes_padded_rank": ab["total_padded_rank"],
        "hbm_gbs_delta": ab["total"] / (d_us * 1e-6) / 1e9 if d_us else None,
        "frac_of_8tbs_delta": ab["total"] / (d_us * 1e-6) / 1e9 / NOMINAL_HBM_GBS if d_us else None,
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s",
                     "duration": ("mean event time of %s alone: a replay of the same steps with "
                                  "the path forced to it, which then does the same work (it "
                                  "takes every active row)" % kernel) if dom_us else
                                 "mean event time of the lora_delta call (its CUDA-core and "
                                 "tensor-core launches together: both have rows)",
                     "frac": achieved / peak if achieved else None, "traffic": traffic},
        "e2e": {"value": w.M / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": K * launches_per_step,
        "launches_per_step": launches_per_step,
        "clocks": clk,
        "wall_s_timed": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
