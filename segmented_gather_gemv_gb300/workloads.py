"""Seeded synthetic inputs for the multi-LoRA delta path.

This module only draws inputs: per-token adapter ids, activations, adapter
pools, base outputs, ranks and scales.  It holds none of the method's
arithmetic, imports neither the CUDA binding nor the oracle, and is the one
module both sides share.

Every workload draws from ``numpy.random.default_rng(seed)`` in a fixed order
(stated per function).  Values are drawn in float32; workloads computed in
bf16 have every floating-point input rounded to bf16 (round to nearest even)
and are returned as float32 arrays that hold those exact bf16 values.

Shapes follow the serving scenarios the LoRA pages describe: a decode batch
of single-token sequences with adapters spread over a pool (the decode SGMV
case of the "vLLM-Ascend LoRA" article, section 3.3), prefill sequences whose
rows share one adapter each (section 3.4), mixed-rank pools padded to the
maximum rank (sections 2.1 and 3.4), a mixed prefill + decode step with a
fused QKV projection split into output slices, and the toy shape of the
"09. Triton Fused LoRA" tutorial's test.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

SEED = 42


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even).

    Returns float32 holding exactly representable bf16 values.  NaN stays
    NaN; no input here is near the float32 overflow limit."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    out = rounded.view(np.float32).copy()
    nan = np.isnan(a)
    if nan.any():
        out[nan] = np.float32("nan")
    return out


@dataclass
class Workload:
    """One batch of inputs for the delta path.

    ids      int32 [M]               adapter slot per token row, -1 = none
    x        float32 [M, d_in]       activations
    A        float32 [n, r_max, d_in]            shrink pool
    B        list of float32 [n, d_out_t, r_max] expand pool per output slice
    y        float32 [M, sum(d_out_t)]           base output (updated in place)
    scale    float                    uniform scale when adapter_scale is None
    adapter_scale  float32 [n] or None (per-adapter alpha / r_a)
    ranks    int32 [n] or None        true rank per adapter (None = r_max)
    """
    name: str
    dtype: str
    ids: np.ndarray
    x: np.ndarray
    A: np.ndarray
    B: List[np.ndarray]
    y: np.ndarray
    scale: float = 1.0
    adapter_scale: Optional[np.ndarray] = None
    ranks: Optional[np.ndarray] = None
    chunk_size: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def M(self) -> int:
        return int(self.ids.shape[0])

    @property
    def d_in(self) -> int:
        return int(self.x.shape[1])

    @property
    def n_adapters(self) -> int:
        return int(self.A.shape[0])

    @property
    def r_max(self) -> int:
        return int(self.A.shape[1])

    @property
    def d_outs(self) -> List[int]:
        return [int(b.shape[1]) for b in self.B]

    @property
    def d_out(self) -> int:
        return int(sum(self.d_outs))

    def with_chunk(self, chunk_size: int) -> "Workload":
        w = Workload(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        w.chunk_size = int(chunk_size)
        w.name = "%s_chunk%d" % (self.name, chunk_size)
        return w


def _normal(rng, shape, std, dtype_name):
    v = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return round_bf16(v) if dtype_name == "bf16" else v


def _zipf_ids(rng, n_pool: int, s: float, size: int) -> np.ndarray:
    """Truncated Zipf law over slots 0..n_pool-1: P(slot k-1) ~ k^-s."""
    k = np.arange(1, n_pool + 1, dtype=np.float64)
    p = k ** (-s)
    p /= p.sum()
    return rng.choice(n_pool, size=size, p=p).astype(np.int32)


def _pad_ranks(A: np.ndarray, Bs: List[np.ndarray], ranks: np.ndarray,
               pad_value: float) -> None:
    for a, r in enumerate(ranks):
        A[a, r:, :] = pad_value
        for B in Bs:
            B[a, :, r:] = pad_value


def page1_toy(seed: int = SEED) -> Workload:
    """The "09. Triton Fused LoRA" test shape: 4 tokens, 128 -> 256, a pool
    of 3 adapters of rank 16, ids [2, 0, 1, 2], fp32, scale 1, base y = 0.

    Draw order: x, A, B (standard normal)."""
    rng = np.random.default_rng(seed)
    M, d_in, d_out, n, r = 4, 128, 256, 3, 16
    x = _normal(rng, (M, d_in), 1.0, "f32")
    A = _normal(rng, (n, r, d_in), 1.0, "f32")
    B = _normal(rng, (n, d_out, r), 1.0, "f32")
    ids = np.array([2, 0, 1, 2], np.int32)
    y = np.zeros((M, d_out), np.float32)
    return Workload("page1_toy", "f32", ids, x, A, [B], y, scale=1.0)


def segment_example(seed: int = SEED) -> Workload:
    """The segment example of "III.Punica: Multi-Tenant LoRA Serving"
    (section SGMV): 7 tokens with ids 2 2 2 5 5 1 1 over a pool of 6
    adapters; fp32, 128 -> 256, rank 16, scale 1, base y standard normal.

    Draw order: x, A, B, y."""
    rng = np.random.default_rng(seed)
    M, d_in, d_out, n, r = 7, 128, 256, 6, 16
    x = _normal(rng, (M, d_in), 1.0, "f32")
    A = _normal(rng, (n, r, d_in), 1.0 / np.sqrt(d_in), "f32")
    B = _normal(rng, (n, d_out, r), 1.0 / np.sqrt(r), "f32")
    y = _normal(rng, (M, d_out), 1.0, "f32")
    ids = np.array([2, 2, 2, 5, 5, 1, 1], np.int32)
    return Workload("segment_example", "f32", ids, x, A, [B], y, scale=1.0)


def decode(seed: int = SEED, M: int = 256, d_in: int = 4096, d_out: int = 4096,
           n_pool: int = 64, n_active: int = 32, r: int = 16,
           alpha: float = 32.0, dtype: str = "bf16") -> Workload:
    """Decode SGMV batch: one token per sequence, ids uniform over
    ``n_active`` adapters drawn without replacement from a pool of
    ``n_pool``; rows in random order (unsorted).

    Draw order: active set, ids, x ~ N(0,1), A ~ N(0, 1/d_in),
    B ~ N(0, 1/r), y ~ N(0,1).  scale = alpha / r."""
    rng = np.random.default_rng(seed)
    active = rng.choice(n_pool, size=n_active, replace=False).astype(np.int32)
    ids = active[rng.integers(0, n_active, size=M)].astype(np.int32)
    x = _normal(rng, (M, d_in), 1.0, dtype)
    A = _normal(rng, (n_pool, r, d_in), 1.0 / np.sqrt(d_in), dtype)
    B = _normal(rng, (n_pool, d_out, r), 1.0 / np.sqrt(r), dtype)
    y = _normal(rng, (M, d_out), 1.0, dtype)
    return Workload("decode_M%d_%dx%d_r%d" % (M, d_in, d_out, r), dtype, ids,
                    x, A, [B], y, scale=alpha / r,
                    meta={"n_active": n_active})


def prefill(seed: int = SEED, n_seq: int = 16, len_lo: int = 128,
            len_hi: int = 1024, n_pool: int = 100, zipf_s: float = 1.1,
            d_in: int = 4096, d_out: int = 4096, r: int = 16,
            alpha: float = 32.0, chunk_size: int = 0,
            dtype: str = "bf16") -> Workload:
    """Prefill batch: ``n_seq`` sequences with lengths uniform in
    [len_lo, len_hi], each on one adapter drawn Zipf(zipf_s) from the pool;
    rows contiguous per sequence, sequences in order.

    Draw order: lengths, adapters, x, A, B, y."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(len_lo, len_hi + 1, size=n_seq)
    seq_ids = _zipf_ids(rng, n_pool, zipf_s, n_seq)
    ids = np.repeat(seq_ids, lens).astype(np.int32)
    M = int(ids.shape[0])
    x = _normal(rng, (M, d_in), 1.0, dtype)
    A = _normal(rng, (n_pool, r, d_in), 1.0 / np.sqrt(d_in), dtype)
    B = _normal(rng, (n_pool, d_out, r), 1.0 / np.sqrt(r), dtype)
    y = _normal(rng, (M, d_out), 1.0, dtype)
    return Workload("prefill_%dseq_M%d_%dx%d_r%d" % (n_seq, M, d_in, d_out, r),
                    dtype, ids, x, A, [B], y, scale=alpha / r,
                    chunk_size=chunk_size,
                    meta={"seq_lens": lens.tolist(), "seq_adapters": seq_ids.tolist()})


MIXED_RANKS = (8, 16, 32, 64)


def mixed_rank(seed: int = SEED, proj: str = "up", M: int = 512,
               n_pool: int = 100, n_active: int = 48, skip_frac: float = 0.25,
               alpha: float = 32.0, pad_value: float = 0.0,
               d_model: int = 4096, d_ff: int = 14336,
               dtype: str = "bf16") -> Workload:
    """Mixed-rank MLP decode batch: ranks per adapter drawn from
    {8, 16, 32, 64}, pool padded to rank 64 (padding = ``pad_value``; NaN in
    the poison tests), ids uniform over ``n_active`` adapters, a fraction
    ``skip_frac`` of the rows set to -1.  ``proj`` "up" (also the gate
    shape) is d_model -> d_ff, "down" is d_ff -> d_model.
    scale_a = alpha / r_a.

    Draw order: ranks, active set, ids, skipped rows, x, A, B, y."""
    if proj not in ("up", "gate", "down"):
        raise ValueError(proj)
    d_in, d_out = (d_model, d_ff) if proj != "down" else (d_ff, d_model)
    rng = np.random.default_rng(seed)
    r_max = max(MIXED_RANKS)
    ranks = np.asarray(MIXED_RANKS, np.int32)[rng.integers(0, len(MIXED_RANKS), size=n_pool)]
    active = rng.choice(n_pool, size=n_active, replace=False).astype(np.int32)
    ids = active[rng.integers(0, n_active, size=M)].astype(np.int32)
    skipped = rng.choice(M, size=int(round(M * skip_frac)), replace=False)
    ids[skipped] = -1
    x = _normal(rng, (M, d_in), 1.0, dtype)
    A = _normal(rng, (n_pool, r_max, d_in), 1.0 / np.sqrt(d_in), dtype)
    B = rng.standard_normal((n_pool, d_out, r_max), dtype=np.float32)
    B *= (1.0 / np.sqrt(ranks.astype(np.float32)))[:, None, None]
    if dtype == "bf16":
        B = round_bf16(B)
    y = _normal(rng, (M, d_out), 1.0, dtype)
    _pad_ranks(A, [B], ranks, pad_value)
    adapter_scale = (np.float32(alpha) / ranks.astype(np.float32)).astype(np.float32)
    return Workload("mixed_rank_%s_M%d_%dx%d" % (proj, M, d_in, d_out), dtype,
                    ids, x, A, [B], y, scale=1.0, adapter_scale=adapter_scale,
                    ranks=ranks, meta={"proj": proj, "pad_value": pad_value})


def _rescale_lengths(lens: np.ndarray, total: int, lo: int, hi: int) -> np.ndarray:
    """Scale integer lengths to sum to ``total`` with every length kept in
    [lo, hi]; the remainder is spread one row at a time from the first
    sequence on."""
    n = lens.shape[0]
    if not (n * lo <= total <= n * hi):
        raise ValueError("total out of reach")
    out = np.clip(np.floor(lens * (total / lens.sum())).astype(np.int64), lo, hi)
    i = 0
    while out.sum() != total:
        step = 1 if out.sum() < total else -1
        if lo <= out[i % n] + step <= hi:
            out[i % n] += step
        i += 1
    return out


def mixed_serving(seed: int = SEED, n_prefill_seq: int = 6,
                  prefill_rows: int = 1536, len_lo: int = 64, len_hi: int = 512,
                  n_decode: int = 512, n_pool: int = 128, zipf_s: float = 1.1,
                  r: int = 32, alpha: float = 64.0, d_in: int = 4096,
                  d_outs=(4096, 1024, 1024), dtype: str = "bf16") -> Workload:
    """Mixed serving step: ``n_prefill_seq`` prefill sequences (lengths
    uniform in [len_lo, len_hi], rescaled to sum to ``prefill_rows``),
    contiguous and first, then ``n_decode`` single-token rows.  Every
    sequence draws its adapter Zipf(zipf_s) from a pool of ``n_pool``.  The
    output is a fused QKV projection: one shared A pool, one B pool per
    output slice (q, k, v), written side by side into y's columns.

    Draw order: lengths, prefill adapters, decode adapters, x, A,
    B (q, k, v), y."""
    rng = np.random.default_rng(seed)
    lens = _rescale_lengths(rng.integers(len_lo, len_hi + 1, size=n_prefill_seq),
                            prefill_rows, len_lo, len_hi)
    pre_ids = _zipf_ids(rng, n_pool, zipf_s, n_prefill_seq)
    dec_ids = _zipf_ids(rng, n_pool, zipf_s, n_decode)
    ids = np.concatenate([np.repeat(pre_ids, lens), dec_ids]).astype(np.int32)
    M = int(ids.shape[0])
    x = _normal(rng, (M, d_in), 1.0, dtype)
    A = _normal(rng, (n_pool, r, d_in), 1.0 / np.sqrt(d_in), dtype)
    Bs = [_normal(rng, (n_pool, d, r), 1.0 / np.sqrt(r), dtype) for d in d_outs]
    y = _normal(rng, (M, int(sum(d_outs))), 1.0, dtype)
    return Workload("mixed_serving_M%d_qkv%d" % (M, sum(d_outs)), dtype, ids, x,
                    A, Bs, y, scale=alpha / r,
                    meta={"seq_lens": lens.tolist(), "n_decode": n_decode})


def random_batch(seed: int, M: int, d_in: int, d_outs, n_pool: int, r_max: int,
                 dtype: str = "bf16", ranks=None, n_active: Optional[int] = None,
                 skip_frac: float = 0.0, bad_frac: float = 0.0,
                 run_len: int = 1, chunk_size: int = 0, scale: float = 0.5,
                 per_adapter_scale: bool = False, pad_value: float = 0.0,
                 y_zero: bool = False) -> Workload:
    """General small batch for parity and edge-case tests.

    ids: ``n_active`` adapters (default: all of the pool) drawn without
    replacement; rows come in runs of ``run_len`` equal ids (run_len > 1
    makes prefill-like contiguous segments); then ``skip_frac`` of the rows
    become -1 and ``bad_frac`` become out-of-range ids (n_pool + k).
    ``ranks`` may be None (uniform r_max), a sequence to draw from per
    adapter, or an explicit per-adapter array.

    Draw order: ranks, active set, run ids, skipped rows, bad rows, x, A, B
    (per slice), y, per-adapter scales."""
    rng = np.random.default_rng(seed)
    d_outs = [int(d) for d in (d_outs if isinstance(d_outs, (list, tuple)) else [d_outs])]
    rk = None
    if ranks is not None:
        ranks = np.asarray(ranks, np.int32)
        if ranks.shape[0] == n_pool:
            rk = ranks.copy()
        else:
            rk = ranks[rng.integers(0, ranks.shape[0], size=n_pool)].astype(np.int32)
    n_active = n_pool if n_active is None else n_active
    active = rng.choice(n_pool, size=n_active, replace=False).astype(np.int32)
    n_runs = (M + run_len - 1) // run_len if M > 0 else 0
    run_ids = active[rng.integers(0, n_active, size=n_runs)] if n_runs else np.zeros(0, np.int32)
    ids = np.repeat(run_ids, run_len)[:M].astype(np.int32)
    if M and skip_frac > 0:
        ids[rng.choice(M, size=int(round(M * skip_frac)), replace=False)] = -1
    if M and bad_frac > 0:
        bad = rng.choice(M, size=max(1, int(round(M * bad_frac))), replace=False)
        ids[bad] = n_pool + rng.integers(0, 7, size=bad.shape[0]).astype(np.int32)
    x = _normal(rng, (M, d_in), 1.0, dtype)
    A = _normal(rng, (n_pool, r_max, d_in), 1.0 / np.sqrt(d_in), dtype)
    Bs = [_normal(rng, (n_pool, d, r_max), 1.0 / np.sqrt(r_max), dtype) for d in d_outs]
    y = (np.zeros((M, sum(d_outs)), np.float32) if y_zero
         else _normal(rng, (M, sum(d_outs)), 1.0, dtype))
    adapter_scale = None
    if per_adapter_scale:
        adapter_scale = rng.uniform(0.25, 2.0, size=n_pool).astype(np.float32)
    if rk is not None:
        _pad_ranks(A, Bs, rk, pad_value)
    name = "random_M%d_%dx%s_n%d_r%d" % (M, d_in, "+".join(map(str, d_outs)), n_pool, r_max)
    return Workload(name, dtype, ids, x, A, Bs, y, scale=scale,
                    adapter_scale=adapter_scale, ranks=rk, chunk_size=chunk_size)


def serving_workloads() -> dict:
    """The five serving scenarios at full size (name -> factory)."""
    return {
        "page1_toy": page1_toy,
        "segment_example": segment_example,
        "decode": decode,
        "prefill": prefill,
        "prefill_chunk64": lambda: prefill(chunk_size=64),
        "mixed_rank_up": lambda: mixed_rank(proj="up"),
        "mixed_rank_down": lambda: mixed_rank(proj="down"),
        "mixed_serving": mixed_serving,
    }
