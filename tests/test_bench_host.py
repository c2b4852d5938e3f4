"""Host-side logic of bench.py (no GPU): the algorithmic byte count behind
roofline.achieved, and the rule that ties committed ncu traffic figures to
the kernel source they were taken on."""
import json
import os

import numpy as np

import bench
from segmented_gather_gemv_gb300 import workloads as wl


def test_decode_algorithmic_bytes_closed_form():
    # 256 rows, 4096 -> 4096, rank 16, bf16, 32 touched adapters:
    # x 256*4096*2, A and B 32*16*4096*2 each, y read + write 2*256*4096*2
    ab = bench.algorithmic_bytes(wl.decode())
    assert ab["active_rows"] == 256 and ab["touched_adapters"] == 32
    assert ab["x"] == 256 * 4096 * 2
    assert ab["A"] == ab["B"] == 32 * 16 * 4096 * 2
    assert ab["y_rw"] == 2 * 256 * 4096 * 2
    assert ab["total"] == 14680064 == ab["total_padded_rank"]


def test_mixed_rank_bytes_use_true_ranks():
    w = wl.mixed_rank(proj="up")
    ab = bench.algorithmic_bytes(w)
    act = (w.ids >= 0) & (w.ids < w.n_adapters)
    touched = np.unique(w.ids[act])
    r_sum = int(w.ranks[touched].sum())
    assert ab["A"] == r_sum * w.d_in * 2 and ab["B"] == r_sum * w.d_out * 2
    assert ab["active_rows"] == int(act.sum())
    assert ab["total"] < ab["total_padded_rank"]  # padding to rank 64 is not counted


def test_whole_job_tokens_per_s():
    assert bench.whole_job_tokens_per_s(1, 10, 256, 1.0) == 2.56e6
    assert bench.whole_job_tokens_per_s(4, 10, 256, 1.0) == 4 * 2.56e6


def test_committed_traffic_follows_the_source(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("// kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"k": ["k.cu"]})
    (tmp_path / "profiles").mkdir()
    h = bench.source_hash("k")
    (tmp_path / "profiles" / "traffic.json").write_text(
        json.dumps({"k": {"w": {"dram_bytes_per_launch": 123, "source_sha256_16": h}}}))
    assert bench.committed_traffic("k", "w") == 123
    assert bench.committed_traffic("k", "other") is None
    src.write_text("// kernel v2\n")  # the kernel changed since the capture
    assert bench.source_hash("k") != h
    assert bench.committed_traffic("k", "w") is None

