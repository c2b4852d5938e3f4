"""CPU oracle for the multi-LoRA delta path -- TEST INFRASTRUCTURE ONLY.

A plain fp64 statement of what the path computes (``lora_oracle.c``), with a
ctypes wrapper.  Only the test suite, the smoke check and the CPU-baseline
leg of ``bench.py`` may import this package.  The product library never
imports it, and it shares no code with the CUDA path: the two meet only in
the seeded input generator, which holds none of the method's arithmetic.

Functions (each cites the passage it follows in ``lora_oracle.c``):

``prepare_batch``  grouping of tokens by adapter (first-appearance order,
                   ascending rows inside a group, optional fixed chunks,
                   id -1 skipped) -- "III.Punica: Multi-Tenant LoRA
                   Serving", sections SGMV and 代码.
``shrink``         h = x . A_id^T per token, true rank only.
``expand``         y += s_id * h . B_id^T per token and output slice.
``delta``          shrink then expand, one token at a time -- the loop of
                   the "09. Triton Fused LoRA" tutorial's test, with the
                   unmerged scaling of the "vLLM-Ascend LoRA" article,
                   section 1.1.

All floating-point inputs are passed as float32 arrays holding the exact
values the GPU sees (bf16 values are exactly representable in float32);
the C code widens every element to double.  Outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liblora_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with plain gcc (no fast-math, no target flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp]
    # OpenMP shares the rows of delta_parallel out over host threads; without
    # it that function runs on one thread (same result either way)
    if subprocess.run(cmd[:1] + ["-fopenmp"] + cmd[1:], capture_output=True).returncode != 0:
        subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32p = ctypes.POINTER(ctypes.c_int32)
            lib.oracle_prepare_batch.restype = ctypes.c_int
            lib.oracle_prepare_batch.argtypes = [
                i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                i32p, i32p, i32p, i32p, i32p]
            lib.oracle_prepare_batch_ordered.restype = ctypes.c_int
            lib.oracle_prepare_batch_ordered.argtypes = [
                i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                i32p, i32p, i32p, i32p, i32p]
            for fn in (lib.oracle_shrink, lib.oracle_expand, lib.oracle_delta,
                       lib.oracle_delta_parallel):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f32(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.float32:
        a = a.astype(np.float32)
    return np.ascontiguousarray(a)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def prepare_batch(ids, n_adapters: int, chunk_size: int = 0, ascending: bool = False) -> dict:
    """Segment metadata for a batch of per-token adapter ids: groups in
    first-appearance order, or by increasing adapter id with ``ascending``.

    Returns a dict with ``sorted_token_ids``, ``seg_indptr``, ``seg_lens``,
    ``weight_indices`` (trimmed to their true lengths) and ``num_segs``,
    ``num_active``, ``num_invalid``.
    """
    lib = _load()
    ids = _i32(ids).reshape(-1)
    M = ids.shape[0]
    cap = max(M, 1)
    sorted_ids = np.zeros(cap, np.int32)
    indptr = np.zeros(cap + 1, np.int32)
    lens = np.zeros(cap, np.int32)
    widx = np.zeros(cap, np.int32)
    counts = np.zeros(3, np.int32)
    rc = lib.oracle_prepare_batch_ordered(
        _ptr(ids, ctypes.c_int32), M, int(n_adapters), int(chunk_size), 1 if ascending else 0,
        _ptr(sorted_ids, ctypes.c_int32), _ptr(indptr, ctypes.c_int32),
        _ptr(lens, ctypes.c_int32), _ptr(widx, ctypes.c_int32),
        _ptr(counts, ctypes.c_int32))
    if rc != 0:
        raise ValueError("oracle_prepare_batch rejected its arguments")
    S, act, bad = (int(v) for v in counts)
    return {
        "sorted_token_ids": sorted_ids[:act].copy(),
        "seg_indptr": indptr[:S + 1].copy(),
        "seg_lens": lens[:S].copy(),
        "weight_indices": widx[:S].copy(),
        "num_segs": S,
        "num_active": act,
        "num_invalid": bad,
    }


class _Slices:
    """Marshals a list of B pools (one per output slice) for the C code."""

    def __init__(self, B_pools):
        self.pools = [_f32(b) for b in B_pools]
        for b in self.pools:
            if b.ndim != 3:
                raise ValueError("each B pool must be (n_adapters, d_out, r_max)")
        n = len(self.pools)
        self.ptrs = (ctypes.POINTER(ctypes.c_float) * n)(
            *[_ptr(b, ctypes.c_float) for b in self.pools])
        self.s_adapter = np.array([b.shape[1] * b.shape[2] for b in self.pools], np.int64)
        self.s_n = np.array([b.shape[2] for b in self.pools], np.int64)
        self.d_out = np.array([b.shape[1] for b in self.pools], np.int32)
        self.col_off = np.zeros(n, np.int32)
        if n > 1:
            self.col_off[1:] = np.cumsum(self.d_out)[:-1]
        self.total = int(self.d_out.sum())
        self.n = n


def _scale_args(scale, adapter_scale):
    if adapter_scale is None:
        return float(scale), None
    return float(scale), np.ascontiguousarray(np.asarray(adapter_scale, np.float64))


def shrink(x, ids, A_pool, ranks=None) -> np.ndarray:
    """h[i, j] = sum_k x[i, k] A[id_i, j, k] for j < r_id (fp64, (M, r_max)).

    Rows without a valid adapter are returned as NaN (undefined)."""
    lib = _load()
    x = _f32(x)
    ids = _i32(ids).reshape(-1)
    A = _f32(A_pool)
    M, d_in = x.shape
    n, r_max, d_in_a = A.shape
    assert d_in_a == d_in and ids.shape[0] == M
    rk = None if ranks is None else _i32(ranks)
    h = np.full((M, r_max), np.nan, np.float64)
    rc = lib.oracle_shrink(
        ctypes.c_int32(M), ctypes.c_int32(d_in), ctypes.c_int32(r_max),
        _ptr(x, ctypes.c_float), ctypes.c_int64(d_in), _ptr(ids, ctypes.c_int32),
        ctypes.c_int32(n), _ptr(A, ctypes.c_float),
        ctypes.c_int64(r_max * d_in), ctypes.c_int64(d_in),
        _ptr(rk, ctypes.c_int32), _ptr(h, ctypes.c_double), ctypes.c_int64(r_max))
    if rc != 0:
        raise ValueError("oracle_shrink rejected its arguments")
    return h


def expand(h, ids, B_pools, y_base, scale=1.0, adapter_scale=None,
           ranks=None) -> np.ndarray:
    """y = y_base + s_id * h . B_id^T over all slices (fp64 result).

    ``B_pools`` is one (n, d_out, r_max) array or a list of them (output
    slices written side by side into y's columns)."""
    lib = _load()
    if not isinstance(B_pools, (list, tuple)):
        B_pools = [B_pools]
    sl = _Slices(B_pools)
    h = np.ascontiguousarray(np.asarray(h, np.float64))
    ids = _i32(ids).reshape(-1)
    M, r_max = h.shape
    n = sl.pools[0].shape[0]
    y = np.array(y_base, dtype=np.float64, copy=True).reshape(M, sl.total)
    rk = None if ranks is None else _i32(ranks)
    sc, asc = _scale_args(scale, adapter_scale)
    rc = lib.oracle_expand(
        ctypes.c_int32(M), ctypes.c_int32(r_max), _ptr(h, ctypes.c_double),
        ctypes.c_int64(r_max), _ptr(ids, ctypes.c_int32), ctypes.c_int32(n),
        _ptr(rk, ctypes.c_int32), ctypes.c_double(sc), _ptr(asc, ctypes.c_double),
        ctypes.c_int32(sl.n), sl.ptrs, _ptr(sl.s_adapter, ctypes.c_int64),
        _ptr(sl.s_n, ctypes.c_int64), _ptr(sl.d_out, ctypes.c_int32),
        _ptr(sl.col_off, ctypes.c_int32), _ptr(y, ctypes.c_double),
        ctypes.c_int64(sl.total))
    if rc != 0:
        raise ValueError("oracle_expand rejected its arguments")
    return y


def delta(x, ids, A_pool, B_pools, y_base, scale=1.0, adapter_scale=None,
          ranks=None, return_h=False, threads=1):
    """y = y_base + s_id (x_i . A_id^T) . B_id^T, token by token (fp64).

    ``threads`` > 1 shares the token rows out over that many host threads
    (``oracle_delta_parallel``: the same per-row arithmetic, bit-identical
    result); the number of threads used is then in ``delta.last_threads``.

    ``A_pool`` may be a list with one pool per output slice (a fused
    projection whose slices each have their own A): slice t's columns then
    get s_id (x_i . A_t[id]^T) . B_t[id]^T, computed by this same per-token
    routine on that slice alone (the slices write disjoint columns)."""
    if isinstance(A_pool, (list, tuple)):
        if not isinstance(B_pools, (list, tuple)):
            B_pools = [B_pools]
        assert len(A_pool) == len(B_pools) and not return_h
        y = np.array(y_base, dtype=np.float64, copy=True)
        col = 0
        for A_t, B_t in zip(A_pool, B_pools):
            d = B_t.shape[1]
            y[:, col:col + d] = delta(x, ids, A_t, [B_t], y[:, col:col + d], scale=scale,
                                      adapter_scale=adapter_scale, ranks=ranks, threads=threads)
            col += d
        return y
    lib = _load()
    if not isinstance(B_pools, (list, tuple)):
        B_pools = [B_pools]
    sl = _Slices(B_pools)
    x = _f32(x)
    ids = _i32(ids).reshape(-1)
    A = _f32(A_pool)
    M, d_in = x.shape
    n, r_max, d_in_a = A.shape
    assert d_in_a == d_in and ids.shape[0] == M
    for b in sl.pools:
        assert b.shape[0] == n and b.shape[2] == r_max
    y = np.array(y_base, dtype=np.float64, copy=True).reshape(M, sl.total)
    rk = None if ranks is None else _i32(ranks)
    sc, asc = _scale_args(scale, adapter_scale)
    if threads > 1 and not return_h:
        used = ctypes.c_int32(0)
        rc = lib.oracle_delta_parallel(
            ctypes.c_int32(M), ctypes.c_int32(d_in), ctypes.c_int32(r_max),
            _ptr(x, ctypes.c_float), ctypes.c_int64(d_in), _ptr(ids, ctypes.c_int32),
            ctypes.c_int32(n), _ptr(A, ctypes.c_float),
            ctypes.c_int64(r_max * d_in), ctypes.c_int64(d_in),
            _ptr(rk, ctypes.c_int32), ctypes.c_double(sc), _ptr(asc, ctypes.c_double),
            ctypes.c_int32(sl.n), sl.ptrs, _ptr(sl.s_adapter, ctypes.c_int64),
            _ptr(sl.s_n, ctypes.c_int64), _ptr(sl.d_out, ctypes.c_int32),
            _ptr(sl.col_off, ctypes.c_int32), _ptr(y, ctypes.c_double),
            ctypes.c_int64(sl.total), ctypes.c_int32(int(threads)), ctypes.byref(used))
        if rc != 0:
            raise ValueError("oracle_delta_parallel rejected its arguments")
        delta.last_threads = int(used.value)
        return y
    delta.last_threads = 1
    h = np.full((M, r_max), np.nan, np.float64) if return_h else None
    rc = lib.oracle_delta(
        ctypes.c_int32(M), ctypes.c_int32(d_in), ctypes.c_int32(r_max),
        _ptr(x, ctypes.c_float), ctypes.c_int64(d_in), _ptr(ids, ctypes.c_int32),
        ctypes.c_int32(n), _ptr(A, ctypes.c_float),
        ctypes.c_int64(r_max * d_in), ctypes.c_int64(d_in),
        _ptr(rk, ctypes.c_int32), ctypes.c_double(sc), _ptr(asc, ctypes.c_double),
        ctypes.c_int32(sl.n), sl.ptrs, _ptr(sl.s_adapter, ctypes.c_int64),
        _ptr(sl.s_n, ctypes.c_int64), _ptr(sl.d_out, ctypes.c_int32),
        _ptr(sl.col_off, ctypes.c_int32), _ptr(y, ctypes.c_double),
        ctypes.c_int64(sl.total), _ptr(h, ctypes.c_double), ctypes.c_int64(r_max))
    if rc != 0:
        raise ValueError("oracle_delta rejected its arguments")
    return (y, h) if return_h else y
