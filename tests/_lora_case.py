"""Test helpers: move a seeded workload to the GPU, run the oracle on the
same rounded values, and compare."""
import numpy as np
import torch

import oracle

# Tolerances on max|y_gpu - y_ref| / max|y_ref - y_base| (the same ratio for h):
# fp32 inputs with fp32 accumulation, and bf16 inputs with fp32 accumulation.
TOL = {"f32": 1e-5, "bf16": 1e-2}
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def to_dev(w, device="cuda"):
    dt = TORCH_DT[w.dtype]
    d = {
        "ids": torch.from_numpy(w.ids).to(device),
        "x": torch.from_numpy(w.x).to(device=device, dtype=dt),
        "A": torch.from_numpy(w.A).to(device=device, dtype=dt),
        "B": [torch.from_numpy(b).to(device=device, dtype=dt) for b in w.B],
        "y": torch.from_numpy(w.y).to(device=device, dtype=dt),
        "ranks": None if w.ranks is None else torch.from_numpy(w.ranks).to(device),
        "adapter_scale": None if w.adapter_scale is None else torch.from_numpy(w.adapter_scale).to(device),
    }
    return d


def oracle_delta(w, return_h=False):
    return oracle.delta(w.x, w.ids, w.A, w.B, w.y, scale=w.scale,
                        adapter_scale=w.adapter_scale, ranks=w.ranks, return_h=return_h)


def rel_err(got, ref, base, rows=None):
    got = np.asarray(got, np.float64)
    if rows is not None:
        got, ref, base = got[rows], ref[rows], base[rows]
    if ref.size == 0:
        return 0.0
    den = np.abs(ref - base).max()
    num = np.abs(got - ref).max()
    if den == 0:
        return 0.0 if num == 0 else float("inf")
    return num / den


def active_rows(w):
    return (w.ids >= 0) & (w.ids < w.n_adapters)
