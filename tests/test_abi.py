"""The C-ABI library builds for sm_103a, loads, exports every symbol the
header declares, and rejects bad arguments on the host (no GPU needed:
argument checks run before any CUDA call)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(lora_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from segmented_gather_gemv_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("lora_workspace_size", "lora_prepare_batch", "lora_shrink", "lora_expand",
              "lora_delta", "lora_last_error_string", "lora_abi_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in sorted(_declared_functions()):
        assert hasattr(lib, n), n


def test_ordered_prepare_rejects_unknown_order(lib):
    # checked on the host before anything is enqueued
    from segmented_gather_gemv_gb300 import binding as B
    raw = B._Batch()
    st = lib.lora_prepare_batch_ordered(None, 4, 4, 0, 0, 7, None, ctypes.c_size_t(0), ctypes.byref(raw), None)
    assert st == B.LORA_ERR_INVALID


def test_workspace_size_host_only(lib):
    f = lib.lora_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int32] * 3
    assert f(256, 64, 0) > 256 * 4
    assert f(9000, 100, 64) > f(9000, 100, 0)
    assert f(0, 1, 0) > 0
    assert f(-1, 4, 0) == 0 and f(4, 0, 0) == 0 and f(4, 4, -2) == 0


def test_bad_arguments_rejected_before_any_cuda_call():
    from segmented_gather_gemv_gb300 import binding as B
    L = B.lib()
    raw = B._Batch()
    st = L.lora_prepare_batch(None, -5, 4, 0, 0, None, 0, ctypes.byref(raw), None)
    assert st == B.LORA_ERR_INVALID
    assert b"M" in L.lora_last_error_string()
    st = L.lora_prepare_batch(None, 4, 4, 0, 0, None, 0, ctypes.byref(raw), None)
    assert st == B.LORA_ERR_INVALID  # ids NULL
    # a batch that lora_prepare_batch never filled
    st = L.lora_delta(ctypes.byref(raw), B.BF16, None, 0, 64, None, 0, 0, 16, None, 1, None,
                      ctypes.c_float(1.0), None, None, 0, 0, None)
    assert st == B.LORA_ERR_INVALID
    assert L.lora_abi_version() == 200
