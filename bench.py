#!/usr/bin/env python
"""Throughput of the multi-LoRA delta path on one GB300 (or N, weak scaling).

One step = one pass of the whole path over one batch of synthetic input:
``lora_prepare_batch`` (device-side grouping) + ``lora_delta`` (fused shrink,
scale and expand), both through the C ABI.  Default workload: the decode
SGMV batch (256 single-token rows, 4096 -> 4096, rank 16, 32 of 64 pool
adapters active, bf16).

Timing: W eager warm-up steps, then exactly K steps captured in CUDA graphs
and replayed between CUDA events on the launching stream, bracketed by a
barrier and a device synchronize.  A GPU-side delay is enqueued just before
the start event, so that the host has submitted the graphs before the start
event runs and the region times the device, not the submission.  Every step
uses one of S rotating input sets (x, y, pools, ids, workspace) whose total
exceeds L2, so no step finds its inputs in L2.  The kernels of a step are
chained by programmatic dependent launch.

Roofline: the dominant kernel is the one the library reports for the delta
call (``lora_last_kernels``); when one kernel takes every active row the path
is forced to it.  Its average launch duration comes from a chain of G
back-to-back ``lora_delta`` calls (prepared batches, rotating input sets)
replayed between CUDA events on the launching stream: the time of the chain
over G.  Per-kernel event times of single launches are reported beside it.

The other serving workloads are measured in the same run (fewer steps, the
same rules) under ``other_workloads``.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
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
    "sgmv_small_kernel": ["segmented_gather_gemv_gb300/csrc/sgmv_small.cu",
                          "segmented_gather_gemv_gb300/csrc/common.cuh"],
    "sgmv_stream_kernel": ["segmented_gather_gemv_gb300/csrc/sgmv_stream.cu",
                           "segmented_gather_gemv_gb300/csrc/common.cuh"],
    "sgmv_cc_kernel": ["segmented_gather_gemv_gb300/csrc/sgmv_cc.cu",
                       "segmented_gather_gemv_gb300/csrc/common.cuh"],
    "sgmv_tc_kernel": ["segmented_gather_gemv_gb300/csrc/sgmv_tc.cu",
                       "segmented_gather_gemv_gb300/csrc/common.cuh"],
}
# Device delay before a timed region: longer than the host needs to submit
# the region's graphs (cycles at about 2 GHz).
DELAY_CYCLES = 4_000_000


def parse_args(argv=None):
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
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads")
    ap.add_argument("--extra-steps", type=int, default=500)
    ap.add_argument("--b-layout", choices=["rank_contiguous", "rank_major"], default="rank_contiguous",
                    help="B pools [n][d_out][r_max] or [n][r_max][d_out] (main workload only)")
    return ap.parse_args(argv)


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


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k = line.split(":")[0].strip().lower()
                if k in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


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
    repeated for about `seconds`, once on all host cores (the rows shared
    out by OpenMP) and once single-threaded."""
    import oracle

    def run(threads, budget):
        t0 = time.perf_counter()
        reps, used = 0, 1
        while True:
            oracle.prepare_batch(w.ids, w.n_adapters, w.chunk_size)
            oracle.delta(w.x, w.ids, w.A, w.B, w.y, scale=w.scale,
                         adapter_scale=w.adapter_scale, ranks=w.ranks, threads=threads)
            used = oracle.delta.last_threads
            reps += 1
            if time.perf_counter() - t0 >= budget:
                break
        dt = time.perf_counter() - t0
        return reps * w.M / dt, reps, dt, used

    cores = host_cores()
    v_all, reps_all, dt_all, used = run(cores, seconds / 2)
    v_one, reps_one, dt_one, _ = run(1, seconds / 2)
    return {"value": v_all, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": "%d full batches of %d rows (grouping + fp64 per-token delta, rows over %d "
                      "threads), %.1f s" % (reps_all, w.M, used, dt_all),
            "cpu_model": cpu_model(), "nproc": cores,
            "single_thread": {"value": v_one, "unit": "tokens/s", "cores": 1,
                              "sample": "%d full batches, %.1f s" % (reps_one, dt_one)}}


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
    cores = host_cores()
    # Per step: a bounded sample of the batch's rows, sized so the whole run
    # takes about two minutes at most.
    t0 = time.perf_counter()
    oracle.delta(w.x[:64], w.ids[:64], w.A, w.B, w.y[:64], scale=w.scale,
                 adapter_scale=w.adapter_scale, ranks=w.ranks, threads=cores)
    per_row = max((time.perf_counter() - t0) / 64, 1e-6)
    rows = int(max(1, min(w.M, 100.0 / (K + W) / per_row)))
    sel = np.arange(rows)

    def step():
        oracle.prepare_batch(w.ids[sel], w.n_adapters, w.chunk_size)
        oracle.delta(w.x[sel], w.ids[sel], w.A, w.B, w.y[sel], scale=w.scale,
                     adapter_scale=w.adapter_scale, ranks=w.ranks, threads=cores)

    for _ in range(W):
        step()
    t0 = time.perf_counter()
    for _ in range(K):
        step()
    dt = time.perf_counter() - t0
    used = oracle.delta.last_threads
    value = K * rows / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": 1e3 * dt / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "tokens_per_step": rows,
                   "sample": "first %d of %d rows per step" % (rows, w.M)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "sample": "first %d of %d rows of %s per step, %d steps, rows over %d "
                                   "threads" % (rows, w.M, w.name, K, used),
                         "cpu_model": cpu_model(), "nproc": cores},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU side

class Bench:
    """Input sets, graphs and timings of one workload on one GPU."""

    def __init__(self, w: wl.Workload, args, dev, stream, path: int, rank_major: bool = False):
        import torch
        from segmented_gather_gemv_gb300 import binding as B
        self.torch, self.B = torch, B
        self.w, self.args, self.dev, self.stream, self.path = w, args, dev, stream, path
        self.es = 2 if w.dtype == "bf16" else 4
        self.tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        # Rotating input sets: enough copies that the sets together exceed L2.
        self.set_bytes = (w.x.size + w.y.size + w.A.size + sum(b.size for b in w.B)) * self.es
        self.n_sets = int(min(64, max(2, math.ceil(3 * L2_BYTES / self.set_bytes))))
        x0 = torch.from_numpy(w.x).to(dev, self.tdt)
        y0 = torch.from_numpy(w.y).to(dev, self.tdt)
        A0 = torch.from_numpy(w.A).to(dev, self.tdt)
        # rank-major B pools, (n, r_max, d_out): an adapter reads only its rank's rows
        self.rank_major = rank_major
        B0 = [torch.from_numpy(b).to(dev, self.tdt) for b in w.B]
        if rank_major:
            B0 = [b.transpose(1, 2).contiguous() for b in B0]
        ids0 = torch.from_numpy(w.ids).to(dev)
        self.ranks = None if w.ranks is None else torch.from_numpy(w.ranks).to(dev)
        self.ascale = None if w.adapter_scale is None else torch.from_numpy(w.adapter_scale).to(dev)
        ws_bytes = B.lora_workspace_size(w.M, w.n_adapters, w.chunk_size)
        self.sets = []
        for i in range(self.n_sets):
            self.sets.append({
                "x": x0 if i == 0 else x0.clone(), "y": y0 if i == 0 else y0.clone(),
                "A": A0 if i == 0 else A0.clone(), "B": B0 if i == 0 else [b.clone() for b in B0],
                "ids": ids0 if i == 0 else ids0.clone(),
                "ws": torch.empty(ws_bytes, dtype=torch.uint8, device=dev),
            })

    def prepare(self, s):
        return self.B.lora_prepare_batch(s["ids"], self.w.n_adapters, self.w.chunk_size,
                                         workspace=s["ws"], stream=self.stream)

    def delta(self, batch, s, path=None):
        self.B.lora_delta(batch, s["x"], s["A"], s["B"], s["y"], scale=self.w.scale, b_rank_major=self.rank_major,
                          adapter_scale=self.ascale, ranks=self.ranks,
                          path=self.path if path is None else path, stream=self.stream)

    def step(self, s):
        batch = self.prepare(s)
        self.delta(batch, s)
        return batch

    def delay(self):
        self.torch.cuda._sleep(DELAY_CYCLES)

    def graph(self, nsteps, offset=0, event_nodes=False):
        """Graph of `nsteps` steps; with `event_nodes`, events bracket every
        kernel (they also cut the programmatic overlap between kernels)."""
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True))
               for _ in range(nsteps if event_nodes else 0)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream, capture_error_mode="thread_local"):
            for i in range(nsteps):
                s = self.sets[(offset + i) % self.n_sets]
                if event_nodes:
                    evs[i][0].record(self.stream)
                batch = self.prepare(s)
                if event_nodes:
                    evs[i][1].record(self.stream)
                self.delta(batch, s)
                if event_nodes:
                    evs[i][2].record(self.stream)
        return g, evs

    def timed(self, graphs, world, dev):
        """Device time of replaying `graphs` (ms), max over ranks."""
        torch = self.torch
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            self.delay()
            t0.record(self.stream)
            for g in graphs:
                g.replay()
            t1.record(self.stream)
        t1.synchronize()
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        return max_over_ranks(t0.elapsed_time(t1), world, dev)

    def incremental_us(self, G, k_rows):
        """Device time (us per step) of G steps that patch k_rows rows of a
        kept batch (lora_batch_update) and then run the delta, against G steps
        that rebuild the batch (lora_prepare_batch) and run the delta, and G
        steps that run the delta on a kept batch whose ids did not change."""
        torch, B, w = self.torch, self.B, self.w
        gen = torch.Generator(device="cpu").manual_seed(5)
        rows = [torch.randperm(w.M, generator=gen)[:k_rows].to(torch.int32).to(self.dev) for _ in range(G)]
        new = [torch.randint(-1, w.n_adapters, (k_rows,), generator=gen).to(torch.int32).to(self.dev)
               for _ in range(G)]
        batches = [self.prepare(s) for s in self.sets]
        with torch.cuda.stream(self.stream):
            for i, b in enumerate(batches):  # the first update copies the ids into the batch
                B.lora_batch_update(b, rows[0], new[0], stream=self.stream)
                self.delta(b, self.sets[i])
        self.stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream, capture_error_mode="thread_local"):
            for i in range(G):
                j = i % self.n_sets
                B.lora_batch_update(batches[j], rows[i], new[i], stream=self.stream)
                self.delta(batches[j], self.sets[j])
        g_full, _ = self.graph(G)
        out = {}
        for name, gr in (("update_step_us", g), ("prepare_step_us", g_full)):
            with torch.cuda.stream(self.stream):
                gr.replay()
            self.stream.synchronize()
            out[name] = 1e3 * self.timed([gr], 1, self.dev) / G
        out["rows_changed_per_step"] = k_rows
        out["update_launches_per_step"] = 2
        # ids unchanged: the kept batch needs neither update nor rebuild
        out["kept_batch_step_us"] = self.delta_chain_us(G, self.path)
        return out

    def split_calls_us(self, G):
        """Device time (us per call) of lora_shrink and of lora_expand, each in
        a chain of G back-to-back calls on prepared batches: the two halves of
        the fused delta, with h in global memory between them."""
        torch, B, w = self.torch, self.B, self.w
        batches = [self.prepare(s) for s in self.sets]
        hs = [torch.zeros((w.M, w.r_max), dtype=torch.float32, device=self.dev) for _ in range(min(self.n_sets, 4))]

        def shrink(i):
            s = self.sets[i % self.n_sets]
            B.lora_shrink(batches[i % self.n_sets], s["x"], s["A"], h=hs[i % len(hs)], ranks=self.ranks,
                          path=self.path, stream=self.stream)

        def expand(i):
            s = self.sets[i % self.n_sets]
            B.lora_expand(batches[i % self.n_sets], hs[i % len(hs)], s["B"], s["y"], scale=w.scale,
                          adapter_scale=self.ascale, ranks=self.ranks, path=self.path, stream=self.stream)

        out = {}
        for name, fn in (("shrink", shrink), ("expand", expand)):
            with torch.cuda.stream(self.stream):
                for i in range(3):
                    fn(i)
            self.stream.synchronize()
            used = B.lora_last_kernels()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream, capture_error_mode="thread_local"):
                for i in range(G):
                    fn(i)
            with torch.cuda.stream(self.stream):
                g.replay()
            self.stream.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(self.stream):
                self.delay()
                e0.record(self.stream)
                g.replay()
                e1.record(self.stream)
            e1.synchronize()
            out[name + "_us"] = 1e3 * e0.elapsed_time(e1) / G
            out[name + "_kernels"] = [n for bit, n in sorted(B.KERNEL_NAMES.items()) if used & bit]
        return out

    def delta_chain_us(self, G, path):
        """Average launch time (us) of lora_delta in a chain of G back-to-back
        calls on prepared batches of the rotating sets."""
        torch = self.torch
        batches = []
        for s in self.sets:
            batches.append(self.prepare(s))
        self.stream.synchronize()
        with torch.cuda.stream(self.stream):
            for i in range(3):
                self.delta(batches[i % self.n_sets], self.sets[i % self.n_sets], path)
        self.stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream, capture_error_mode="thread_local"):
            for i in range(G):
                self.delta(batches[i % self.n_sets], self.sets[i % self.n_sets], path)
        with torch.cuda.stream(self.stream):
            g.replay()
        self.stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            self.delay()
            e0.record(self.stream)
            g.replay()
            e1.record(self.stream)
        e1.synchronize()
        return 1e3 * e0.elapsed_time(e1) / G


def measure(b: Bench, key: str, K: int, W: int, world: int, dev, graph_steps: int, clocks=None,
            kernel_events=True) -> dict:
    """One workload: W warm-up steps, K timed steps, the dominant kernel's
    average launch time and the roofline."""
    torch, B, w = b.torch, b.B, b.w
    ab = algorithmic_bytes(w)
    with torch.cuda.stream(b.stream):
        for i in range(W):
            b.step(b.sets[i % b.n_sets])
    b.stream.synchronize()
    b0 = b.prepare(b.sets[0])
    b.stream.synchronize()
    counts = b0.counts()
    n_launch0 = B.lora_launch_count()
    with torch.cuda.stream(b.stream):
        batch = b.prepare(b.sets[0])
        b.delta(batch, b.sets[0])
    kernels_bits = B.lora_last_kernels()
    launches_per_step = B.lora_launch_count() - n_launch0
    b.stream.synchronize()

    # The dominant kernel: the only one of the delta call, or, when one
    # kernel takes every active row, the path forced to it.
    dom_path, dom_bits = None, kernels_bits
    if bin(kernels_bits).count("1") > 1 and b.path == 0 and counts["num_active"] > 0:
        if counts["tc_rows"] == counts["num_active"]:
            dom_path = 2
        elif counts["tc_rows"] == 0:
            dom_path = 1
        if dom_path is not None:
            with torch.cuda.stream(b.stream):
                b.delta(b0, b.sets[0], dom_path)
            dom_bits = B.lora_last_kernels()
            b.stream.synchronize()
    kernel = (B.KERNEL_NAMES.get(dom_bits) if bin(dom_bits).count("1") == 1
              else "+".join(B.KERNEL_NAMES[k] for k in sorted(B.KERNEL_NAMES) if dom_bits & k))

    G = max(1, min(graph_steps, K))
    reps, rem = divmod(K, G)
    g_main, _ = b.graph(G)
    g_rem = b.graph(rem)[0] if rem else None
    with torch.cuda.stream(b.stream):
        g_main.replay()
        if g_rem is not None:
            g_rem.replay()
    b.stream.synchronize()
    graphs = [g_main] * reps + ([g_rem] if g_rem is not None else [])
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
    wall0 = time.perf_counter()
    elapsed_ms = b.timed(graphs, world, dev)
    wall = time.perf_counter() - wall0
    clk = clocks.stop() if clocks is not None else None

    # the dominant kernel's average launch time (a chain of delta calls)
    Gc = max(32, min(512, K))
    chain_us = b.delta_chain_us(Gc, dom_path)
    # single launches with event nodes around each kernel, for context
    kern = {}
    if kernel_events:
        Ge = min(64, max(8, K))
        g_ev, evs = b.graph(Ge, event_nodes=True)
        with torch.cuda.stream(b.stream):
            g_ev.replay()
            g_ev.replay()
        b.stream.synchronize()
        prep = [1e3 * e0.elapsed_time(e1) for e0, e1, e2 in evs]
        dlt = [1e3 * e1.elapsed_time(e2) for e0, e1, e2 in evs]
        kern = {"prepare_single_launch_mean": statistics.mean(prep),
                "delta_single_launch_mean": statistics.mean(dlt)}
    kern["delta_chain_mean"] = chain_us

    peak, peak_kind = load_peaks()
    achieved = ab["total"] / (chain_us * 1e-6) / 1e9
    ms_per_step = elapsed_ms / K
    out = {
        "workload": w.name, "steps": K, "warmup": W, "ms_per_step": ms_per_step,
        "value": whole_job_tokens_per_s(world, K, w.M, elapsed_ms), "elapsed_ms": elapsed_ms,
        "wall_s_timed": wall, "counts": counts, "ab": ab, "launches_per_step": launches_per_step,
        "n_sets": b.n_sets, "graph_steps": G, "clocks": clk,
        "kernels_us": kern,
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
                     "duration": ("mean launch time of %s in a chain of %d back-to-back lora_delta "
                                  "calls%s (CUDA events on the launching stream around the chain)"
                                  % (kernel, Gc, " with the path forced to it" if dom_path else "")),
                     "traffic": committed_traffic(kernel, key) if kernel in KERNEL_SOURCES else None},
        "step_gbs": ab["total"] / (ms_per_step * 1e-3) / 1e9,
    }
    return out


def e2e_measure(b: Bench, steps: int) -> dict:
    """The public API from pinned host buffers, copies inside the timed region.

    Every step copies its inputs in (x, y, ids), runs prepare + delta and
    copies its result (y) out.  The steps run as a serving loop runs them:
    captured in a CUDA graph, device buffer sets in rotation, the input copies
    of later steps (x and ids on one stream, y on another) and the output copy
    of the step before beside a step's kernels.  A buffer set is refilled only
    after the output copy of its previous step has finished."""
    torch, w = b.torch, b.w
    x_h = torch.from_numpy(w.x).to(b.tdt).pin_memory()
    y_h = torch.from_numpy(w.y).to(b.tdt).pin_memory()
    ids_h = torch.from_numpy(w.ids).pin_memory()
    y_out = torch.empty_like(y_h).pin_memory()
    nb = min(3, len(b.sets))
    comp = b.stream
    s_x, s_y, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_x = [torch.cuda.Event() for _ in range(nb)]
    ev_y = [torch.cuda.Event() for _ in range(nb)]
    ev_c = [torch.cuda.Event() for _ in range(nb)]
    ev_o = [torch.cuda.Event() for _ in range(nb)]
    G = max(1, min(16, steps))
    reps = max(1, (steps + G - 1) // G)

    def one(i):
        k = i % nb
        s = b.sets[k]
        with torch.cuda.stream(s_x):
            if i >= nb:
                s_x.wait_event(ev_o[k])
            s["x"].copy_(x_h, non_blocking=True)
            s["ids"].copy_(ids_h, non_blocking=True)
            ev_x[k].record(s_x)
        with torch.cuda.stream(s_y):
            if i >= nb:
                s_y.wait_event(ev_o[k])
            s["y"].copy_(y_h, non_blocking=True)
            ev_y[k].record(s_y)
        comp.wait_event(ev_x[k])
        comp.wait_event(ev_y[k])
        b.step(s)
        ev_c[k].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c[k])
            y_out.copy_(s["y"], non_blocking=True)
            ev_o[k].record(s_out)

    # eager warm-up (also builds the batches' host state), then the graph
    with torch.cuda.stream(comp):
        for i in range(nb):
            root = torch.cuda.Event()
            root.record(comp)
            for st in (s_x, s_y, s_out):
                st.wait_event(root)
            one(i)
            tail = torch.cuda.Event()
            tail.record(s_out)
            comp.wait_event(tail)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=comp):
        root = torch.cuda.Event()
        root.record(comp)
        for st in (s_x, s_y, s_out):
            st.wait_event(root)
        for i in range(G):
            one(i)
        for st in (s_x, s_y, s_out):
            j = torch.cuda.Event()
            j.record(st)
            comp.wait_event(j)
    with torch.cuda.stream(comp):
        g.replay()
    comp.synchronize()
    e_a = torch.cuda.Event(enable_timing=True)
    e_b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(comp):
        e_a.record(comp)
        for _ in range(reps):
            g.replay()
        e_b.record(comp)
    e_b.synchronize()
    e2e_ms = e_a.elapsed_time(e_b) / (reps * G)
    h2d = (x_h.numel() + y_h.numel()) * b.es + ids_h.numel() * 4
    d2h = y_out.numel() * b.es
    return {"value": w.M / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}


def summary(m: dict) -> dict:
    r = m["roofline"]
    return {"workload": m["workload"], "tokens_per_s": m["value"], "ms_per_step": m["ms_per_step"],
            "steps": m["steps"], "algorithmic_bytes_per_step": m["ab"]["total"],
            "step_gbs": m["step_gbs"], "kernel": r["kernel"], "kernel_chain_us": m["kernels_us"]["delta_chain_mean"],
            "roofline_frac": r["frac"], "frac_of_8tbs": r["frac_of_8tbs"], "traffic": r["traffic"],
            "tc_rows": m["counts"]["tc_rows"], "active_rows": m["counts"]["num_active"],
            "num_segs": m["counts"]["num_segs"]}


def run_ours(args, rank: int, world: int, local_rank: int):
    import torch

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    factory, default_steps = WORKLOADS[args.workload]
    K = args.steps if args.steps is not None else default_steps
    W = max(3, args.warmup)
    w = factory(replica_seed(rank))
    stream = torch.cuda.Stream(device=dev)
    b = Bench(w, args, dev, stream, args.path, rank_major=args.b_layout == "rank_major")

    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    clocks = ClockSampler(vis.split(",")[local_rank].strip() if vis else str(local_rank))
    m = measure(b, args.workload + ("+rank_major" if b.rank_major else ""), K, W, world, dev, args.graph_steps,
                clocks=clocks)
    e2e = e2e_measure(b, args.e2e_steps)
    incremental = None
    if args.path == 0 and w.M <= 2048 and world == 1:
        # a decode step that keeps its grouping and patches the rows that
        # changed (a few sequences join or leave), against the full rebuild
        incremental = b.incremental_us(min(256, max(8, K)), max(1, w.M // 32))
    split_calls = None
    if world == 1 and not b.rank_major:
        # the same batch through lora_shrink then lora_expand (h in global memory)
        split_calls = b.split_calls_us(min(64, max(8, K)))
    del b
    torch.cuda.empty_cache()

    others = {}
    if not args.no_extras and args.path == 0:
        for name, (fac, _) in WORKLOADS.items():
            if name == args.workload:
                continue
            wo = fac(replica_seed(rank))
            # the padded mixed-rank pools in the rank-major layout, which reads
            # only each adapter's rank rows
            rm = name.startswith("mixed_rank")
            bo = Bench(wo, args, dev, stream, 0, rank_major=rm)
            mo = measure(bo, name + ("+rank_major" if rm else ""), args.extra_steps, W, world, dev,
                         args.graph_steps, kernel_events=False)
            others[name] = summary(mo)
            others[name]["b_layout"] = "rank_major" if rm else "rank_contiguous"
            del bo
            torch.cuda.empty_cache()

    if rank != 0:
        return
    ab, r = m["ab"], m["roofline"]
    line = {
        "metric": METRIC, "value": m["value"], "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": m["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {
            "workload": w.name, "tokens_per_step": w.M, "active_rows": ab["active_rows"],
            "touched_adapters": ab["touched_adapters"], "num_segs": m["counts"]["num_segs"],
            "chunk_size": w.chunk_size, "path": ["auto", "cuda_core", "tensor"][args.path],
            "b_layout": args.b_layout,
            "l2": "inputs rotate over %d sets (%.0f MB > %d MB L2)"
                  % (m["n_sets"], m["n_sets"] * b_set_bytes(w) / 1e6, L2_BYTES // 2**20),
            "timing": ("CUDA graphs of %d steps (kernels chained by programmatic dependent launch), "
                       "a device-side delay before the start event so the host's submission is "
                       "not timed" % m["graph_steps"]),
            "parallelism": "replicas: one independent batch per GPU" if world > 1 else "single GPU",
        },
        "kernels_us": m["kernels_us"],
        "algorithmic_bytes_per_step": ab["total"],
        "algorithmic_bytes_padded_rank": ab["total_padded_rank"],
        "step_gbs": m["step_gbs"],
        "step_frac_of_8tbs": m["step_gbs"] / NOMINAL_HBM_GBS,
        "roofline": {k: r[k] for k in ("bound", "kernel", "achieved", "peak", "peak_kind", "unit",
                                      "frac", "traffic", "duration")},
        "e2e": {k: e2e[k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step",
                                   "ms_per_step")},
        "gpu_launches": K * m["launches_per_step"],
        "launches_per_step": m["launches_per_step"],
        "clocks": m["clocks"],
        "wall_s_timed": m["wall_s_timed"],
    }
    if incremental is not None:
        line["incremental_grouping"] = incremental
    if split_calls is not None:
        line["split_calls"] = split_calls
    if others:
        line["other_workloads"] = others
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def b_set_bytes(w: wl.Workload) -> int:
    es = 2 if w.dtype == "bf16" else 4
    return (w.x.size + w.y.size + w.A.size + sum(b.size for b in w.B)) * es


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
