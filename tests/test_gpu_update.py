"""Incremental grouping cache: lora_batch_update patches a prepared batch
when rows join, leave or switch adapters ("vLLM-Ascend LoRA" article,
sections 4.2 and 5.3); after a seeded sequence of updates the deltas match
the oracle on the patched ids, and the refreshed metadata matches
oracle.prepare_batch on them bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemv_gb300 import workloads as wl
from tests._lora_case import TOL, active_rows, oracle_delta, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from segmented_gather_gemv_gb300 import binding
    binding.lib()
    return binding


def _arrays_match(batch, ids, n, chunk):
    got = batch.arrays()
    ref = oracle.prepare_batch(ids, n, chunk)
    assert got["num_segs"] == ref["num_segs"]
    assert got["num_active"] == ref["num_active"]
    assert got["num_invalid"] == ref["num_invalid"]
    for k in ("sorted_token_ids", "seg_indptr", "seg_lens", "weight_indices"):
        assert np.array_equal(got[k].numpy(), ref[k]), k


def _apply(cur, rows, new):
    for r, v in zip(rows, new):  # in order: a repeated row takes its last value
        cur[r] = v


# (rows, pool, d_in, d_outs, r_max, chunk): a decode batch (single-pass kernel),
# a batch for the streaming kernel, and one above its limit (the kernels that
# read the metadata, rebuilt in the call while the batch is stale)
CASES = [(256, 64, 1024, [768], 16, 0), (1500, 40, 512, [384, 128], 32, 0), (5000, 300, 256, [256], 16, 7)]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_update_sequence(B, ci):
    M, n, d_in, d_outs, r_max, chunk = CASES[ci]
    rng = np.random.default_rng(900 + ci)
    w = wl.random_batch(seed=901 + ci, M=M, d_in=d_in, d_outs=d_outs, n_pool=n, r_max=r_max,
                        dtype="bf16", skip_frac=0.2, chunk_size=chunk)
    cur = w.ids.copy()
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], n, chunk)
    for step in range(6):
        k = int(rng.integers(1, 40))
        rows = rng.choice(M, size=k, replace=False)
        if step % 2 == 1:
            rows = np.concatenate([rows, rows[:1]])  # a row named twice: the later entry wins
        new = rng.integers(-1, n, size=rows.shape[0]).astype(np.int32)  # -1: the row leaves
        _apply(cur, rows, new)
        B.lora_batch_update(batch, torch.from_numpy(rows.astype(np.int32)).cuda(), torch.from_numpy(new).cuda())
        assert batch.raw.stale == 1
        w.ids = cur.copy()
        y = d["y"].clone()
        B.lora_delta(batch, d["x"], d["A"], d["B"], y, scale=w.scale)
        torch.cuda.synchronize()
        yg = y.float().cpu().numpy().astype(np.float64)
        ref = oracle_delta(w)
        act = active_rows(w)
        assert rel_err(yg, ref, w.y.astype(np.float64), act) <= TOL["bf16"]
        assert np.array_equal(yg[~act], w.y[~act].astype(np.float64)), "inactive rows changed"
    # the caller's ids were not touched
    assert np.array_equal(d["ids"].cpu().numpy(), wl.random_batch(
        seed=901 + ci, M=M, d_in=d_in, d_outs=d_outs, n_pool=n, r_max=r_max, dtype="bf16",
        skip_frac=0.2, chunk_size=chunk).ids)
    B.lora_batch_refresh(batch)
    assert batch.raw.stale == 0
    _arrays_match(batch, cur, n, chunk)
    assert batch.counts()["device_error"] == 0


def test_stale_batch_on_a_metadata_path(B):
    # lora_shrink reads the segment metadata: it is rebuilt inside the call
    M, n = 300, 12
    w = wl.random_batch(seed=950, M=M, d_in=256, d_outs=[128], n_pool=n, r_max=16, dtype="bf16")
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], n, 0)
    rows = np.arange(0, M, 7, dtype=np.int32)
    new = ((w.ids[rows] + 5) % n).astype(np.int32)
    B.lora_batch_update(batch, torch.from_numpy(rows).cuda(), torch.from_numpy(new).cuda())
    cur = w.ids.copy()
    cur[rows] = new
    h = torch.full((M, 16), -777.0, device="cuda")
    B.lora_shrink(batch, d["x"], d["A"], h=h)
    torch.cuda.synchronize()
    h_ref = oracle.shrink(w.x, cur, w.A)
    act = (cur >= 0) & (cur < n)
    hg = h.cpu().numpy().astype(np.float64)
    assert np.abs(hg[act] - h_ref[act]).max() / np.abs(h_ref[act]).max() <= TOL["bf16"]
    assert batch.raw.stale == 1  # the call rebuilt the metadata but left the flag
    B.lora_batch_refresh(batch)
    _arrays_match(batch, cur, n, 0)


def test_update_row_out_of_range(B):
    M, n = 64, 8
    w = wl.random_batch(seed=960, M=M, d_in=128, d_outs=[64], n_pool=n, r_max=16, dtype="bf16")
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], n, 0)
    rows = torch.tensor([3, M + 5, -2, 10], dtype=torch.int32, device="cuda")
    new = torch.tensor([1, 2, 3, -1], dtype=torch.int32, device="cuda")
    B.lora_batch_update(batch, rows, new)
    # the counters report it until the metadata is rebuilt
    assert batch.counts()["device_error"] & B.DEVERR_ROW
    B.lora_batch_refresh(batch)
    cur = w.ids.copy()
    cur[3] = 1
    cur[10] = -1
    _arrays_match(batch, cur, n, 0)


def test_update_rejects_bad_arguments(B):
    w = wl.random_batch(seed=970, M=16, d_in=128, d_outs=[64], n_pool=4, r_max=16, dtype="bf16")
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], 4, 0)
    with pytest.raises(ValueError):
        B.lora_batch_update(batch, torch.zeros(3, dtype=torch.int32, device="cuda"),
                            torch.zeros(2, dtype=torch.int32, device="cuda"))
    B.lora_batch_update(batch, torch.zeros(0, dtype=torch.int32, device="cuda"),
                        torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert batch.raw.stale == 0  # nothing to patch
