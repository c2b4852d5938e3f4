"""Thin Python binding of the C ABI in ``include/lora_sgmv.h``.

Argument marshalling only: every step of the path runs in the CUDA library.
PyTorch supplies device memory and the current stream.  The binding raises
if the library has not been built (``segmented_gather_gemv_gb300.build``)
or if a call returns an error status; there is no fallback.

Calls (same names as the C ABI):
  lora_workspace_size(M, n_adapters, chunk_size) -> int
  lora_prepare_batch(ids, n_adapters, chunk_size=0, tc_min_rows=0, order=0) -> Batch
    (calls lora_prepare_batch_ordered)
  lora_prepare_batch_static(ids, n_adapters, chunk_size=0, tc_min_rows=0) -> Batch
  lora_shrink(batch, x, A_pool, h=None, ranks=None, path=PATH_AUTO) -> h
  lora_expand(batch, h, B_pools, y, scale=1.0, adapter_scale=None,
              ranks=None, y_cols=None, path=PATH_AUTO) -> y
  lora_delta(batch, x, A_pool, B_pools, y, scale=1.0, adapter_scale=None,
             ranks=None, y_cols=None, path=PATH_AUTO) -> y
  lora_batch_update(batch, rows, new_ids) -> batch
  lora_batch_refresh(batch) -> batch
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

from . import build as _build

LORA_OK = 0
LORA_ERR_INVALID = -1
LORA_ERR_UNSUPPORTED = -2
LORA_ERR_WORKSPACE = -3
LORA_ERR_CUDA = -4
F32, BF16 = 0, 1
PATH_AUTO, PATH_CUDA_CORE, PATH_TENSOR = 0, 1, 2
LORA_ORDER_FIRST_APPEARANCE, LORA_ORDER_ASCENDING = 0, 1
MAX_SLICES = 4
COUNT_NAMES = ("num_segs", "num_active", "num_invalid", "num_small_segs",
               "num_tc_segs", "tc_rows", "device_error", "num_groups")
DEVERR_RANK, DEVERR_WAIT, DEVERR_ROW = 1, 2, 4
KERNEL_PREPARE, KERNEL_SMALL, KERNEL_CUDA_CORE, KERNEL_TENSOR, KERNEL_STREAM = 1, 2, 4, 8, 16
KERNEL_NAMES = {KERNEL_PREPARE: "prepare_kernel", KERNEL_SMALL: "sgmv_small_kernel",
                KERNEL_CUDA_CORE: "sgmv_cc_kernel", KERNEL_TENSOR: "sgmv_tc_kernel",
                KERNEL_STREAM: "sgmv_stream_kernel"}

_STATUS = {LORA_ERR_INVALID: "invalid argument", LORA_ERR_UNSUPPORTED: "unsupported",
           LORA_ERR_WORKSPACE: "workspace too small", LORA_ERR_CUDA: "CUDA error"}


class LoraError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s (%d): %s" % (_STATUS.get(status, "error"), status, msg))
        self.status = status


class _Batch(ctypes.Structure):
    _fields_ = [("sorted_token_ids", ctypes.c_void_p), ("seg_indptr", ctypes.c_void_p),
                ("seg_lens", ctypes.c_void_p), ("weight_indices", ctypes.c_void_p),
                ("seg_records", ctypes.c_void_p), ("small_segs", ctypes.c_void_p), ("tc_segs", ctypes.c_void_p),
                ("tc_indptr", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("M", ctypes.c_int32), ("n_adapters", ctypes.c_int32),
                ("chunk_size", ctypes.c_int32), ("max_segs", ctypes.c_int32),
                ("tc_min_rows", ctypes.c_int32), ("magic", ctypes.c_uint32),
                ("ids", ctypes.c_void_p), ("ids_store", ctypes.c_void_p),
                ("order", ctypes.c_int32), ("stale", ctypes.c_int32)]


class _BSlice(ctypes.Structure):
    _fields_ = [("B_pool", ctypes.c_void_p), ("stride_adapter", ctypes.c_int64),
                ("stride_n", ctypes.c_int64), ("d_out", ctypes.c_int32),
                ("y_col", ctypes.c_int32), ("A_pool", ctypes.c_void_p), ("stride_r", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    "CUDA library %s is missing: build it with "
                    "`python -m segmented_gather_gemv_gb300.build`" % path)
            L = ctypes.CDLL(path)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            L.lora_workspace_size.restype = ctypes.c_size_t
            L.lora_workspace_size.argtypes = [i32, i32, i32]
            L.lora_prepare_batch.restype = ctypes.c_int
            L.lora_prepare_batch.argtypes = [vp, i32, i32, i32, i32, vp, ctypes.c_size_t,
                                             ctypes.POINTER(_Batch), vp]
            L.lora_prepare_batch_ordered.restype = ctypes.c_int
            L.lora_prepare_batch_ordered.argtypes = [vp, i32, i32, i32, i32, i32, vp, ctypes.c_size_t,
                                                     ctypes.POINTER(_Batch), vp]
            L.lora_prepare_batch_static.restype = ctypes.c_int
            L.lora_prepare_batch_static.argtypes = [vp, i32, i32, i32, i32, ctypes.POINTER(_Batch), vp]
            L.lora_shrink.restype = ctypes.c_int
            L.lora_shrink.argtypes = [ctypes.POINTER(_Batch), i32, vp, i64, i32, vp, i64, i64,
                                      i32, vp, vp, i64, i32, vp]
            L.lora_expand.restype = ctypes.c_int
            L.lora_expand.argtypes = [ctypes.POINTER(_Batch), i32, vp, i64, i32,
                                      ctypes.POINTER(_BSlice), i32, vp, ctypes.c_float, vp, vp,
                                      i64, i32, vp]
            L.lora_delta.restype = ctypes.c_int
            L.lora_delta.argtypes = [ctypes.POINTER(_Batch), i32, vp, i64, i32, vp, i64, i64, i32,
                                     ctypes.POINTER(_BSlice), i32, vp, ctypes.c_float, vp, vp,
                                     i64, i32, vp]
            L.lora_last_error_string.restype = ctypes.c_char_p
            L.lora_last_error_string.argtypes = []
            L.lora_abi_version.restype = ctypes.c_int32
            L.lora_launch_count.restype = ctypes.c_int64
            L.lora_last_kernels.restype = ctypes.c_int32
            L.lora_last_kernels.argtypes = []
            L.lora_batch_update.restype = ctypes.c_int
            L.lora_batch_update.argtypes = [ctypes.POINTER(_Batch), vp, vp, i32, vp]
            L.lora_batch_refresh.restype = ctypes.c_int
            L.lora_batch_refresh.argtypes = [ctypes.POINTER(_Batch), vp]
            L.lora_selftest_wait.restype = ctypes.c_int
            L.lora_selftest_wait.argtypes = [vp, vp]
            _lib = L
    return _lib


def _check(status: int):
    if status != LORA_OK:
        msg = lib().lora_last_error_string().decode(errors="replace")
        raise LoraError(status, msg)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("unsupported dtype %s (float32 or bfloat16)" % t.dtype)


def _dev_ptr(t: Optional[torch.Tensor], what: str, dtype=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % what)
    # the library launches on the current device (and keeps a static
    # workspace per device): tensors of another device would be read across
    if t.device.index != torch.cuda.current_device():
        raise ValueError("%s is on cuda:%d, the current device is cuda:%d"
                         % (what, t.device.index, torch.cuda.current_device()))
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s" % (what, dtype))
    return t.data_ptr()


def _inner_contig(t: torch.Tensor, what: str):
    if t.dim() < 1:
        raise ValueError("%s must have at least one dimension" % what)
    if t.numel() and t.stride(-1) != 1:
        raise ValueError("%s must have a contiguous last dimension" % what)


def _ld(t: torch.Tensor, dim: int = 0) -> int:
    """Row stride of a tensor (the row length when it holds no elements)."""
    if t.numel() == 0:
        n = 1
        for s in t.shape[dim + 1:]:
            n *= s
        return n
    return t.stride(dim)


class _DeviceInts:
    """n int32 at a device address, for torch.as_tensor (no copy)."""

    def __init__(self, ptr: int, n: int):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4", "data": (ptr, False), "version": 3}


class Batch:
    """Device segment metadata of one batch (wraps ``lora_batch_t``).

    Holds a reference to its workspace, which must stay alive while the
    batch is used."""

    def __init__(self, raw: _Batch, workspace: torch.Tensor, ids: torch.Tensor):
        self.raw = raw
        self.workspace = workspace
        self.ids = ids

    @property
    def M(self) -> int:
        return self.raw.M

    @property
    def max_segs(self) -> int:
        return self.raw.max_segs

    def _view(self, field: str, n: int) -> torch.Tensor:
        ptr = getattr(self.raw, field)
        if self.workspace is None:  # the library's own workspace: wrap the device pointer
            return torch.as_tensor(_DeviceInts(ptr, n), device="cuda")
        base = self.workspace.data_ptr()
        off = ptr - base
        assert off % 4 == 0 and off >= 0
        flat = self.workspace.view(torch.int32)
        return flat[off // 4: off // 4 + n]

    def counts(self) -> dict:
        """Device counters (synchronises with the current stream)."""
        c = self._view("counts", len(COUNT_NAMES)).cpu().tolist()
        return dict(zip(COUNT_NAMES, c))

    def arrays(self) -> dict:
        """Copies of the device arrays, trimmed to their valid lengths."""
        c = self.counts()
        S, act = c["num_segs"], c["num_active"]
        return {
            "sorted_token_ids": self._view("sorted_token_ids", act).cpu(),
            "seg_indptr": self._view("seg_indptr", S + 1).cpu(),
            "seg_lens": self._view("seg_lens", S).cpu(),
            "weight_indices": self._view("weight_indices", S).cpu(),
            "seg_records": self._view("seg_records", 32 * self.max_segs).cpu().view(-1, 32),
            "small_segs": self._view("small_segs", 4 * c["num_small_segs"]).cpu().view(-1, 4),
            "tc_segs": self._view("tc_segs", 4 * c["num_tc_segs"]).cpu().view(-1, 4),
            "tc_indptr": self._view("tc_indptr", c["num_tc_segs"] + 1).cpu(),
            **c,
        }


def lora_launch_count() -> int:
    """Kernel launches the library has enqueued in this process."""
    return int(lib().lora_launch_count())


def lora_selftest_wait(counts: torch.Tensor, stream=None) -> None:
    """Run the bounded-wait diagnostic: sets DEVERR_WAIT in counts[6]."""
    if counts.dtype != torch.int32 or not counts.is_cuda or counts.numel() < len(COUNT_NAMES):
        raise ValueError("counts must be a CUDA int32 tensor of %d entries" % len(COUNT_NAMES))
    _check(lib().lora_selftest_wait(ctypes.c_void_p(counts.data_ptr()), ctypes.c_void_p(_stream(stream))))


def lora_batch_update(batch: Batch, rows: torch.Tensor, new_ids: torch.Tensor, stream=None) -> Batch:
    """Row rows[k] now carries adapter new_ids[k] (-1: none), on the device;
    the batch's metadata is rebuilt lazily (lora_batch_refresh)."""
    rows = rows.to(torch.int32).contiguous()
    new_ids = new_ids.to(torch.int32).contiguous()
    if rows.shape != new_ids.shape or rows.dim() != 1:
        raise ValueError("rows and new_ids must be 1-D of the same length")
    n = rows.numel()
    _check(lib().lora_batch_update(ctypes.byref(batch.raw), _dev_ptr(rows, "rows") if n else None,
                                   _dev_ptr(new_ids, "new_ids") if n else None, n, _stream(stream)))
    batch._keep = (rows, new_ids)  # alive until the kernel that reads them has run
    return batch


def lora_batch_refresh(batch: Batch, stream=None) -> Batch:
    """Rebuilds the metadata of a batch whose ids were updated."""
    _check(lib().lora_batch_refresh(ctypes.byref(batch.raw), _stream(stream)))
    return batch


def lora_last_kernels() -> int:
    """Bit set (KERNEL_*) of the kernels the calling thread's last call enqueued."""
    return int(lib().lora_last_kernels())


def lora_workspace_size(M: int, n_adapters: int, chunk_size: int = 0) -> int:
    return int(lib().lora_workspace_size(int(M), int(n_adapters), int(chunk_size)))


def lora_prepare_batch(ids: torch.Tensor, n_adapters: int, chunk_size: int = 0,
                       tc_min_rows: int = 0, workspace: Optional[torch.Tensor] = None,
                       stream=None, order: int = 0) -> Batch:
    """Build segment metadata on the device for per-token adapter ids;
    ``order`` is LORA_ORDER_FIRST_APPEARANCE (default) or
    LORA_ORDER_ASCENDING."""
    if ids.dim() != 1:
        raise ValueError("ids must be 1-D")
    M = ids.shape[0]
    ids_ptr = _dev_ptr(ids, "ids", torch.int32) if M else (ids.data_ptr() or None)
    if M and not ids.is_contiguous():
        raise ValueError("ids must be contiguous")
    need = lora_workspace_size(M, n_adapters, chunk_size)
    if need == 0:
        raise LoraError(LORA_ERR_INVALID, "bad batch size arguments")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=ids.device if M else "cuda")
    ws_ptr = _dev_ptr(workspace, "workspace")
    raw = _Batch()
    _check(lib().lora_prepare_batch_ordered(ids_ptr, M, int(n_adapters), int(chunk_size), int(tc_min_rows),
                                            int(order), ws_ptr,
                                            workspace.numel() * workspace.element_size(),
                                            ctypes.byref(raw), _stream(stream)))
    return Batch(raw, workspace, ids)


def lora_prepare_batch_static(ids: torch.Tensor, n_adapters: int, chunk_size: int = 0,
                              tc_min_rows: int = 0, stream=None) -> Batch:
    """lora_prepare_batch into the library's own device workspace (no
    allocation); the batch is valid until the next call of this function on
    the same device has run."""
    if ids.dim() != 1:
        raise ValueError("ids must be 1-D")
    M = ids.shape[0]
    ids_ptr = _dev_ptr(ids, "ids", torch.int32) if M else (ids.data_ptr() or None)
    if M and not ids.is_contiguous():
        raise ValueError("ids must be contiguous")
    raw = _Batch()
    _check(lib().lora_prepare_batch_static(ids_ptr, M, int(n_adapters), int(chunk_size), int(tc_min_rows),
                                           ctypes.byref(raw), _stream(stream)))
    return Batch(raw, None, ids)


def _slices(B_pools, y: torch.Tensor, y_cols, r_max: int, dtype, rank_major: bool = False):
    if isinstance(B_pools, torch.Tensor):
        B_pools = [B_pools]
    B_pools = list(B_pools)
    if not 1 <= len(B_pools) <= MAX_SLICES:
        raise ValueError("1..%d B pools" % MAX_SLICES)
    arr = (_BSlice * len(B_pools))()
    col = 0
    for t, B in enumerate(B_pools):
        if B.dim() != 3 or B.dtype != dtype:
            raise ValueError("B pool %d must be (n, %s) of the input dtype"
                             % (t, "r_max, d_out" if rank_major else "d_out, r_max"))
        _inner_contig(B, "B pool")
        arr[t].B_pool = _dev_ptr(B, "B pool")
        arr[t].stride_adapter = _ld(B)
        d_out = B.shape[2] if rank_major else B.shape[1]
        if rank_major:  # (n, r_max, d_out): rank rows of d_out outputs
            arr[t].stride_n = 1
            arr[t].stride_r = _ld(B, 1)
        else:
            arr[t].stride_n = _ld(B, 1)
            arr[t].stride_r = 0
        arr[t].d_out = d_out
        arr[t].y_col = int(y_cols[t]) if y_cols is not None else col
        col += d_out
    return arr, len(B_pools)


def _ranks_scale(ranks, adapter_scale):
    rp = _dev_ptr(ranks, "ranks", torch.int32)
    sp = _dev_ptr(adapter_scale, "adapter_scale", torch.float32)
    return rp, sp


def lora_shrink(batch: Batch, x: torch.Tensor, A_pool: torch.Tensor,
                h: Optional[torch.Tensor] = None, ranks: Optional[torch.Tensor] = None,
                path: int = PATH_AUTO, stream=None) -> torch.Tensor:
    """h[i, :r] = x[i] . A[id_i]^T (fp32, unscaled) for rows in a segment."""
    _inner_contig(x, "x")
    _inner_contig(A_pool, "A_pool")
    n, r_max, d_in = A_pool.shape
    if h is None:
        h = torch.zeros((batch.M, r_max), dtype=torch.float32, device=x.device)
    _inner_contig(h, "h")
    rp, _ = _ranks_scale(ranks, None)
    _check(lib().lora_shrink(ctypes.byref(batch.raw), _dtype_code(x), _dev_ptr(x, "x"), _ld(x),
                             d_in, _dev_ptr(A_pool, "A_pool", x.dtype), _ld(A_pool),
                             _ld(A_pool, 1), r_max, rp, _dev_ptr(h, "h", torch.float32),
                             _ld(h), int(path), _stream(stream)))
    return h


def lora_expand(batch: Batch, h: torch.Tensor, B_pools, y: torch.Tensor, scale: float = 1.0,
                adapter_scale: Optional[torch.Tensor] = None,
                ranks: Optional[torch.Tensor] = None, y_cols: Optional[Sequence[int]] = None,
                path: int = PATH_AUTO, stream=None) -> torch.Tensor:
    """y[i, slice] += s_id * h[i] . B_id^T for rows in a segment (in place)."""
    _inner_contig(h, "h")
    _inner_contig(y, "y")
    r_max = (B_pools if isinstance(B_pools, torch.Tensor) else B_pools[0]).shape[2]
    arr, ns = _slices(B_pools, y, y_cols, r_max, y.dtype)
    rp, sp = _ranks_scale(ranks, adapter_scale)
    _check(lib().lora_expand(ctypes.byref(batch.raw), _dtype_code(y), _dev_ptr(h, "h", torch.float32),
                             _ld(h), r_max, arr, ns, rp, float(scale), sp, _dev_ptr(y, "y"),
                             _ld(y), int(path), _stream(stream)))
    return y


def lora_delta(batch: Batch, x: torch.Tensor, A_pool, B_pools, y: torch.Tensor,
               scale: float = 1.0, adapter_scale: Optional[torch.Tensor] = None,
               ranks: Optional[torch.Tensor] = None, y_cols: Optional[Sequence[int]] = None,
               path: int = PATH_AUTO, stream=None, b_rank_major: bool = False) -> torch.Tensor:
    """y[i] += s_id * (x[i] . A_id^T) . B_id^T, fused (in place).

    ``A_pool`` may be a list with one A pool per B pool (each slice of a fused
    projection with its own A; the pools share shape and strides).  With
    ``b_rank_major`` the B pools are (n, r_max, d_out): rank-major."""
    _inner_contig(x, "x")
    A_slices = None
    if isinstance(A_pool, (list, tuple)):
        A_slices = list(A_pool)
        A_pool = A_slices[0]
        for a in A_slices:
            _inner_contig(a, "A_pool")
            if a.shape != A_pool.shape or a.stride() != A_pool.stride():
                raise ValueError("per-slice A pools must share shape and strides")
    _inner_contig(A_pool, "A_pool")
    _inner_contig(y, "y")
    n, r_max, d_in = A_pool.shape
    arr, ns = _slices(B_pools, y, y_cols, r_max, x.dtype, rank_major=b_rank_major)
    if A_slices is not None:
        if len(A_slices) != ns:
            raise ValueError("one A pool per B pool")
        for t, a in enumerate(A_slices):
            arr[t].A_pool = _dev_ptr(a, "A_pool", x.dtype)
    rp, sp = _ranks_scale(ranks, adapter_scale)
    _check(lib().lora_delta(ctypes.byref(batch.raw), _dtype_code(x), _dev_ptr(x, "x"), _ld(x), d_in,
                            _dev_ptr(A_pool, "A_pool", x.dtype), _ld(A_pool), _ld(A_pool, 1),
                            r_max, arr, ns, rp, float(scale), sp, _dev_ptr(y, "y", x.dtype),
                            _ld(y), int(path), _stream(stream)))
    return y
