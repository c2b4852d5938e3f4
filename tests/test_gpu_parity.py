"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.  Segment metadata must match bit for bit; values must
match within max|y - y_ref| / max|y_ref - y_base| <= 1e-5 (fp32 inputs) or
1e-2 (bf16 inputs, fp32 accumulation); rows outside every segment must be
left bit-identical."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemv_gb300 import workloads as wl
from tests._lora_case import TOL, active_rows, oracle_delta, rel_err, to_dev

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def B():
    from segmented_gather_gemv_gb300 import binding
    binding.lib()
    return binding


# ----------------------------------------------------------------- grouping

def _check_prepare(B, ids_np, n, chunk, tc_min=0, ascending=False):
    ids = torch.from_numpy(np.asarray(ids_np, np.int32)).cuda()
    batch = B.lora_prepare_batch(ids, n, chunk, tc_min_rows=tc_min,
                                 order=B.LORA_ORDER_ASCENDING if ascending else B.LORA_ORDER_FIRST_APPEARANCE)
    got = batch.arrays()
    ref = oracle.prepare_batch(ids_np, n, chunk, ascending=ascending)
    assert got["num_segs"] == ref["num_segs"]
    assert got["num_active"] == ref["num_active"]
    assert got["num_invalid"] == ref["num_invalid"]
    for k in ("sorted_token_ids", "seg_indptr", "seg_lens", "weight_indices"):
        assert np.array_equal(got[k].numpy(), ref[k]), k
    # path split: every segment in exactly one list, by its adapter group's rows
    thr = tc_min if tc_min > 0 else batch.raw.tc_min_rows
    lens = ref["seg_lens"]
    ids_a = np.asarray(ids_np, np.int64)
    valid = (ids_a >= 0) & (ids_a < n)
    group_rows = np.bincount(ids_a[valid], minlength=n)
    to_tc = group_rows[ref["weight_indices"]] >= thr
    recs = np.stack([ref["seg_indptr"][:-1], lens, ref["weight_indices"],
                     np.arange(len(lens))], axis=1).astype(np.int32).reshape(-1, 4)
    desc = got["seg_records"].numpy()
    S = len(lens)
    flag = 0x40000000
    assert np.array_equal(desc[:S, :3], recs[:, :3])
    assert np.array_equal(desc[:S, 3] & ~flag, recs[:, 3])
    assert np.array_equal((desc[:S, 3] & flag) != 0, to_tc)
    assert np.all(desc[S:, 1] == 0), "descriptors past the last segment must have len 0"
    for s_ in range(S):
        k = min(int(lens[s_]), 28)
        st = int(ref["seg_indptr"][s_])
        assert np.array_equal(desc[s_, 4:4 + k], ref["sorted_token_ids"][st:st + k])
    assert np.array_equal(got["small_segs"].numpy().reshape(-1, 4), recs[~to_tc])
    assert np.array_equal(got["tc_segs"].numpy().reshape(-1, 4), recs[to_tc])
    big = lens[to_tc]
    assert np.array_equal(got["tc_indptr"].numpy(), np.concatenate([[0], np.cumsum(big)]).astype(np.int32))
    assert got["device_error"] == 0
    return batch


def test_prepare_punica_page_example(B):
    g = json.load(open(os.path.join(GOLDEN, "punica_segment_example.json")))
    batch = _check_prepare(B, g["ids"], g["n_adapters"], 0)
    assert batch.arrays()["seg_indptr"].tolist() == g["seg_indptr"]


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("chunk", [0, 1, 3, 64, 5000])
@pytest.mark.parametrize("M,n", [(1, 1), (7, 6), (256, 64), (2047, 100), (9000, 3000), (20000, 8)])
def test_prepare_bit_exact(B, seed, chunk, M, n):
    rng = np.random.default_rng(seed * 1000 + M)
    ids = rng.integers(-1, n, size=M).astype(np.int32)
    if seed == 1:
        ids = np.repeat(rng.integers(0, n, size=(M + 99) // 100), 100)[:M].astype(np.int32)
    if seed == 2:
        ids[rng.choice(M, size=max(1, M // 10), replace=False)] = n + 5  # out of range
    _check_prepare(B, ids, n, chunk, tc_min=[0, 16, 64, 1][seed])


def test_prepare_ascending_punica_ids(B):
    batch = _check_prepare(B, [2, 2, 2, 5, 5, 1, 1], 6, 0, ascending=True)
    assert batch.arrays()["seg_indptr"].tolist() == [0, 2, 5, 7]
    assert batch.arrays()["weight_indices"].tolist() == [1, 2, 5]


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("chunk", [0, 3, 64])
@pytest.mark.parametrize("M,n", [(7, 6), (256, 64), (2047, 100), (9000, 3000), (20000, 8)])
def test_prepare_ascending_bit_exact(B, seed, chunk, M, n):
    rng = np.random.default_rng(seed * 1000 + M + 7)
    ids = rng.integers(-1, n, size=M).astype(np.int32)
    if seed == 1:
        ids = np.repeat(rng.integers(0, n, size=(M + 99) // 100), 100)[:M].astype(np.int32)
    if seed == 2:
        ids[rng.choice(M, size=max(1, M // 10), replace=False)] = n + 5  # out of range
    _check_prepare(B, ids, n, chunk, tc_min=[0, 16, 64][seed], ascending=True)


def test_prepare_ascending_large_pool(B):
    rng = np.random.default_rng(8)
    _check_prepare(B, rng.integers(0, 200000, size=30000).astype(np.int32), 200000, 0, ascending=True)


@pytest.mark.parametrize("n_decode", [60, 400])
def test_delta_ascending_order(B, n_decode):
    # the delta does not depend on the group order; both kernels take rows
    w = wl.mixed_serving(n_prefill_seq=3, prefill_rows=500, len_lo=64, len_hi=300, n_decode=n_decode,
                         n_pool=24, r=16, d_in=1024, d_outs=(512, 256, 256))
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], w.n_adapters, 0, order=B.LORA_ORDER_ASCENDING)
    assert batch.arrays()["weight_indices"].tolist() == sorted(set(int(a) for a in w.ids if a >= 0))
    y = d["y"]
    B.lora_delta(batch, d["x"], d["A"], d["B"], y, scale=w.scale)
    torch.cuda.synchronize()
    _assert_delta(w, y.float().cpu().numpy().astype(np.float64))
    assert batch.counts()["tc_rows"] > 0 and batch.counts()["device_error"] == 0


def test_prepare_degenerate(B):
    _check_prepare(B, np.zeros(0, np.int32), 4, 0)
    _check_prepare(B, np.full(50, -1, np.int32), 4, 0)
    _check_prepare(B, np.full(50, 3, np.int32), 4, 7)
    _check_prepare(B, np.array([99, -7, 2], np.int32), 4, 0)


def test_prepare_large_pool_and_batch(B):
    rng = np.random.default_rng(7)
    _check_prepare(B, rng.integers(0, 200000, size=30000).astype(np.int32), 200000, 0)
    _check_prepare(B, rng.integers(0, 50, size=70000).astype(np.int32), 50, 96)


def test_prepare_workspace_too_small(B):
    ids = torch.zeros(16, dtype=torch.int32, device="cuda")
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.LoraError) as e:
        B.lora_prepare_batch(ids, 4, 0, workspace=ws)
    assert e.value.status == B.LORA_ERR_WORKSPACE


# ----------------------------------------------------------------- values

def _run_delta(B, w, path=0, tc_min=0, guard_cols=0):
    d = to_dev(w)
    ids = d["ids"]
    batch = B.lora_prepare_batch(ids, w.n_adapters, w.chunk_size, tc_min_rows=tc_min)
    y = d["y"]
    if guard_cols:
        # y inside a wider buffer whose extra columns hold a sentinel
        big = torch.full((w.M, w.d_out + guard_cols), 12345.0, dtype=y.dtype, device="cuda")
        big[:, :w.d_out] = y
        y = big[:, :w.d_out]
    B.lora_delta(batch, d["x"], d["A"], d["B"], y, scale=w.scale, adapter_scale=d["adapter_scale"],
                 ranks=d["ranks"], path=path)
    torch.cuda.synchronize()
    if guard_cols:
        assert torch.all(big[:, w.d_out:] == 12345.0), "write outside y's columns"
    return y.float().cpu().numpy().astype(np.float64), batch


def _assert_delta(w, y_gpu, counts=None):
    y_ref = oracle_delta(w)
    act = active_rows(w)
    err = rel_err(y_gpu, y_ref, w.y.astype(np.float64), act)
    assert err <= TOL[w.dtype], "rel err %.3e > %.0e" % (err, TOL[w.dtype])
    assert np.array_equal(y_gpu[~act], w.y[~act].astype(np.float64)), "inactive rows changed"
    assert np.isfinite(y_gpu).all()
    return err


@pytest.mark.parametrize("path", [0, 1])
def test_page1_toy(B, path):
    w = wl.page1_toy()
    y, _ = _run_delta(B, w, path)
    _assert_delta(w, y)
    assert np.abs(y - oracle_delta(w)).max() < 1e-3  # the page's own criterion


def test_segment_example_values(B):
    w = wl.segment_example()
    y, batch = _run_delta(B, w)
    _assert_delta(w, y)


SMALL_CASES = [
    # several row tiles per segment, ragged d, mixed ranks, slices, skips
    dict(M=300, d_in=1000, d_outs=[776], n_pool=5, r_max=16, run_len=40),
    dict(M=257, d_in=520, d_outs=[264, 64, 136], n_pool=9, r_max=32, ranks=[8, 16, 24, 32],
         skip_frac=0.2, bad_frac=0.05, per_adapter_scale=True),
    dict(M=64, d_in=4096, d_outs=[4096], n_pool=16, r_max=16),
    dict(M=33, d_in=64, d_outs=[128], n_pool=40, r_max=64, ranks=[8, 16, 32, 64], skip_frac=0.25),
    dict(M=90, d_in=2048, d_outs=[512], n_pool=3, r_max=128, run_len=30),
    dict(M=200, d_in=304, d_outs=[96], n_pool=12, r_max=8, ranks=[1, 3, 5, 8], run_len=25),
    dict(M=1, d_in=256, d_outs=[256], n_pool=2, r_max=16),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ci", range(len(SMALL_CASES)))
@pytest.mark.parametrize("chunk", [0, 7])
def test_delta_small(B, dtype, ci, chunk):
    w = wl.random_batch(seed=100 + ci, dtype=dtype, chunk_size=chunk, **SMALL_CASES[ci])
    y, batch = _run_delta(B, w, path=1, guard_cols=8 if dtype == "bf16" else 4)
    _assert_delta(w, y)
    c = batch.counts()
    assert c["num_invalid"] == int(((w.ids >= w.n_adapters) | (w.ids < -1)).sum())
    assert c["device_error"] == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ci", [0, 1, 3])
def test_shrink_and_expand(B, dtype, ci):
    w = wl.random_batch(seed=200 + ci, dtype=dtype, **SMALL_CASES[ci])
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], w.n_adapters, 0)
    guard = torch.full((w.M, w.r_max + 4), -777.0, device="cuda")
    h = guard[:, :w.r_max]
    B.lora_shrink(batch, d["x"], d["A"], h=h, ranks=d["ranks"], path=1)
    torch.cuda.synchronize()
    act = active_rows(w)
    assert torch.all(guard[:, w.r_max:] == -777.0)
    assert torch.all(h[torch.from_numpy(~act).cuda()] == -777.0), "h rows outside segments written"
    h_ref = oracle.shrink(w.x, w.ids, w.A, ranks=w.ranks)
    hg = h.cpu().numpy().astype(np.float64)
    err = np.abs(hg[act] - h_ref[act]).max() / np.abs(h_ref[act]).max()
    assert err <= TOL[dtype]
    # expand from a seeded h of its own (not the GPU's)
    rng = np.random.default_rng(5)
    h_in = rng.standard_normal((w.M, w.r_max)).astype(np.float32)
    y = d["y"].clone()
    B.lora_expand(batch, torch.from_numpy(h_in).cuda(), d["B"], y, scale=w.scale,
                  adapter_scale=d["adapter_scale"], ranks=d["ranks"], path=1)
    y_ref = oracle.expand(h_in, w.ids, w.B, w.y, scale=w.scale, adapter_scale=w.adapter_scale,
                          ranks=w.ranks)
    yg = y.float().cpu().numpy().astype(np.float64)
    assert rel_err(yg, y_ref, w.y.astype(np.float64), act) <= TOL[dtype]
    assert np.array_equal(yg[~act], w.y[~act].astype(np.float64))


def test_mixed_rank_nan_padding_never_read(B):
    w = wl.random_batch(seed=300, M=128, d_in=512, d_outs=[384], n_pool=10, r_max=64,
                        ranks=[8, 16, 32, 64], dtype="bf16", pad_value=float("nan"),
                        per_adapter_scale=True)
    y, _ = _run_delta(B, w, path=1)
    _assert_delta(w, y)


def test_rank_out_of_range_sets_device_error(B):
    w = wl.random_batch(seed=301, M=40, d_in=128, d_outs=[64], n_pool=4, r_max=16, dtype="bf16")
    w.ranks = np.array([16, 99, 16, 16], np.int32)  # adapter 1 claims rank 99 > r_max
    y, batch = _run_delta(B, w, path=1)
    assert batch.counts()["device_error"] & B.DEVERR_RANK
    bad = w.ids == 1
    assert np.array_equal(y[bad], w.y[bad].astype(np.float64))


# Per-adapter ranks with more segments than clusters: the small-segment
# kernel deals its tiles to the clusters by estimated cost (the work plan).
PLAN_CASES = [
    dict(M=600, d_in=4096, d_outs=[2048], n_pool=120, r_max=64, ranks=[8, 16, 32, 64]),       # one tile each
    dict(M=3200, d_in=2048, d_outs=[1024], n_pool=80, r_max=64, ranks=[8, 16, 32, 64], run_len=40),  # several tiles each
    dict(M=700, d_in=2048, d_outs=[1536, 512], n_pool=90, r_max=32, ranks=[8, 16, 24, 32], chunk_size=7,
         skip_frac=0.1, per_adapter_scale=True),                                              # chunks, slices, skips
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("ci", range(len(PLAN_CASES)))
def test_work_plan_mixed_ranks(B, dtype, ci):
    w = wl.random_batch(seed=500 + ci, dtype=dtype, **PLAN_CASES[ci])
    y, batch = _run_delta(B, w, path=1)
    _assert_delta(w, y)
    c = batch.counts()
    assert c["device_error"] == 0 and c["num_segs"] > 38  # more segments than clusters of 4 on 152 SMs


def test_work_plan_rank_out_of_range(B):
    # a bad rank inside a planned batch: flagged, its rows untouched, the rest exact
    w = wl.random_batch(seed=510, M=600, d_in=4096, d_outs=[2048], n_pool=120, r_max=64,
                        ranks=[8, 16, 32, 64], dtype="bf16")
    bad_a = int(w.ids[0])
    w.ranks = w.ranks.copy()
    w.ranks[bad_a] = 99
    y, batch = _run_delta(B, w, path=1)
    assert batch.counts()["device_error"] & B.DEVERR_RANK
    bad = w.ids == bad_a
    assert np.array_equal(y[bad], w.y[bad].astype(np.float64))
    good = wl.Workload(**{**w.__dict__})
    good.ranks = w.ranks.copy()
    good.ranks[bad_a] = 0  # the oracle's view: that adapter adds nothing
    _assert_delta(good, y)


def test_empty_and_all_skipped(B):
    for ids in (np.zeros(0, np.int32), np.full(9, -1, np.int32)):
        w = wl.random_batch(seed=302, M=len(ids), d_in=64, d_outs=[64], n_pool=3, r_max=8, dtype="bf16")
        w.ids = ids
        y, _ = _run_delta(B, w)
        assert np.array_equal(y, w.y.astype(np.float64))


def test_unaligned_pointer_rejected(B):
    w = wl.random_batch(seed=303, M=8, d_in=64, d_outs=[64], n_pool=2, r_max=8, dtype="bf16")
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], 2, 0)
    xb = torch.zeros(8 * 64 + 1, dtype=torch.bfloat16, device="cuda")[1:].view(8, 64)
    with pytest.raises(B.LoraError) as e:
        B.lora_delta(batch, xb, d["A"], d["B"], d["y"])
    assert e.value.status == B.LORA_ERR_UNSUPPORTED


# ------------------------------------------------ full-size serving scenarios

FULL = ["decode", "prefill", "prefill_chunk64", "mixed_rank_up", "mixed_rank_down", "mixed_serving"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_scenarios(B, name):
    w = wl.serving_workloads()[name]()
    y, batch = _run_delta(B, w)
    err = _assert_delta(w, y)
    c = batch.counts()
    assert c["device_error"] == 0
    assert c["num_active"] == int(active_rows(w).sum())
    print("%s: rel err %.3e" % (name, err))


def test_mixed_rank_nan_padding_full_size(B):
    w = wl.mixed_rank(proj="down", pad_value=float("nan"))
    y, _ = _run_delta(B, w)
    _assert_delta(w, y)


def test_large_batch_of_small_groups(B):
    """A batch large enough for a full tensor-core grid whose rows all sit in
    small adapter groups: every segment goes to the CUDA-core kernel, which
    then runs with the smallest cluster count it allows beside that grid."""
    w = wl.random_batch(seed=77, M=10240, d_in=512, d_outs=[384], n_pool=1500, r_max=16,
                        run_len=2, skip_frac=0.05)
    y, batch = _run_delta(B, w)
    c = batch.counts()
    assert c["tc_rows"] == 0 and c["num_small_segs"] > 500
    _assert_delta(w, y)


# ----------------------------------------------------- non-finite base outputs

NONFINITE_CASES = [
    # (workload kwargs, path): every kernel of the path sees NaN and infinities in y
    (dict(M=256, d_in=1024, d_outs=[768], n_pool=40, r_max=16), 0),          # small-batch kernel
    (dict(M=1500, d_in=512, d_outs=[384], n_pool=60, r_max=16), 1),          # small-segment kernel
    (dict(M=700, d_in=512, d_outs=[256, 128], n_pool=6, r_max=16, run_len=120), 2),  # tensor cores only
    (dict(M=900, d_in=512, d_outs=[384], n_pool=30, r_max=32, run_len=40, ranks=[8, 16, 32],
          per_adapter_scale=True), 0),                                        # both kernels
]


@pytest.mark.parametrize("ci", range(len(NONFINITE_CASES)))
def test_nonfinite_y_stays_per_element(B, ci):
    kw, path = NONFINITE_CASES[ci]
    w = wl.random_batch(seed=700 + ci, dtype="bf16", **kw)
    rng = np.random.default_rng(701 + ci)
    act_rows = np.flatnonzero(active_rows(w))
    y = w.y.copy()
    # several non-finite values, some in the same row and 16-column group
    for v in (np.nan, np.inf, -np.inf):
        for _ in range(6):
            i = int(rng.choice(act_rows))
            c = int(rng.integers(0, y.shape[1]))
            y[i, c] = v
            y[i, c ^ 1] = v
    w.y = y
    got, batch = _run_delta(B, w, path=path)
    ref = oracle_delta(w)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "NaN positions differ"
    assert np.array_equal(np.isposinf(got), np.isposinf(ref)), "+inf positions differ"
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), "-inf positions differ"
    act = active_rows(w)
    fin = np.isfinite(ref) & np.isfinite(y) & act[:, None]
    den = np.abs(ref[fin] - y.astype(np.float64)[fin]).max()
    assert np.abs(got[fin] - ref[fin]).max() / den <= TOL["bf16"]
    ok = ~act
    assert np.array_equal(got[ok], y[ok].astype(np.float64), equal_nan=True), "inactive rows changed"
    if path == 2 or ci == 3:
        assert batch.counts()["tc_rows"] > 0


# ------------------------------------------------ the streaming kernel

# Shapes that stream several K and N chunks per tile and several tiles per
# cluster through the streaming kernel: more rows than threads (2, 4 and 8
# rows per thread), projections wider than one stage, per-slice B pools,
# padded ranks, groups of hundreds of rows, and very small d.
PIPE_CASES = [
    dict(M=2048, d_in=4096, d_outs=[4096, 1024, 1024], n_pool=128, r_max=32, run_len=9),
    dict(M=512, d_in=4096, d_outs=[14336], n_pool=100, r_max=64, ranks=[8, 16, 32, 64], skip_frac=0.25),
    dict(M=512, d_in=14336, d_outs=[4096], n_pool=100, r_max=64, ranks=[8, 16, 32, 64], skip_frac=0.25,
         per_adapter_scale=True),
    dict(M=2048, d_in=1024, d_outs=[1024], n_pool=300, r_max=16, run_len=3),
    dict(M=2000, d_in=2048, d_outs=[2048], n_pool=4, r_max=16, run_len=700),
    dict(M=1000, d_in=256, d_outs=[200], n_pool=50, r_max=16, ranks=[1, 3, 5, 8, 16], skip_frac=0.1),
    dict(M=777, d_in=1536, d_outs=[520, 264], n_pool=20, r_max=32, ranks=[8, 16, 24, 32], run_len=30,
         bad_frac=0.05),
]


@pytest.mark.parametrize("ci", range(len(PIPE_CASES)))
def test_stream_kernel_pipeline(B, ci):
    w = wl.random_batch(seed=800 + ci, dtype="bf16", **PIPE_CASES[ci])
    y, batch = _run_delta(B, w, path=1, guard_cols=8)
    assert B.lora_last_kernels() == B.KERNEL_STREAM
    _assert_delta(w, y)
    assert batch.counts()["device_error"] == 0


# ------------------------------------------- split calls at full size

@pytest.mark.parametrize("name", ["decode", "prefill", "prefill_chunk64", "mixed_serving"])
def test_split_calls_full_size(B, name):
    """lora_shrink then lora_expand on the full-size serving configurations:
    h against the oracle's shrink, and the expand (fed the oracle's h, not the
    GPU's) against the oracle's expand; rows outside every segment untouched."""
    w = wl.serving_workloads()[name]()
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], w.n_adapters, w.chunk_size)
    act = active_rows(w)
    guard = torch.full((w.M, w.r_max + 4), -777.0, device="cuda")
    h = guard[:, :w.r_max]
    B.lora_shrink(batch, d["x"], d["A"], h=h, ranks=d["ranks"])
    torch.cuda.synchronize()
    assert torch.all(guard[:, w.r_max:] == -777.0)
    h_ref = oracle.shrink(w.x, w.ids, w.A, ranks=w.ranks)
    hg = h.cpu().numpy().astype(np.float64)
    err = np.abs(hg[act] - h_ref[act]).max() / np.abs(h_ref[act]).max()
    assert err <= TOL[w.dtype], "shrink rel err %.3e" % err
    assert np.all(hg[~act] == -777.0), "h rows outside segments written"
    # the expand from the oracle's h (rounded to fp32), inactive rows zero
    h_in = np.where(act[:, None], h_ref, 0.0).astype(np.float32)
    y = d["y"].clone()
    B.lora_expand(batch, torch.from_numpy(h_in).cuda(), d["B"], y, scale=w.scale,
                  adapter_scale=d["adapter_scale"], ranks=d["ranks"])
    y_ref = oracle.expand(h_in, w.ids, w.B, w.y, scale=w.scale, adapter_scale=w.adapter_scale,
                          ranks=w.ranks)
    yg = y.float().cpu().numpy().astype(np.float64)
    e2 = rel_err(yg, y_ref, w.y.astype(np.float64), act)
    assert e2 <= TOL[w.dtype], "expand rel err %.3e" % e2
    assert np.array_equal(yg[~act], w.y[~act].astype(np.float64))
    assert batch.counts()["device_error"] == 0


# ------------------------------------------------- per-slice A pools

# (workload kwargs, path, kernel): the stacked shrink on the streaming kernel
# (QKV with r 16: 48 stacked ranks; two slices of r 32; a decode-sized batch),
# and one pass per slice where the stacked ranks exceed 64 (decode batch with
# r 32 on the small-batch kernel, rank 64) or the batch exceeds the streaming
# kernel's limit
PER_SLICE_A_CASES = [
    (dict(M=700, d_in=1024, d_outs=[1024, 256, 256], n_pool=40, r_max=16, run_len=20,
          ranks=[8, 16], per_adapter_scale=True, skip_frac=0.1), 0, "sgmv_stream_kernel"),
    (dict(M=1200, d_in=512, d_outs=[384, 128], n_pool=30, r_max=32, ranks=[8, 24, 32]), 1, "sgmv_stream_kernel"),
    (dict(M=200, d_in=1024, d_outs=[512, 256, 256], n_pool=20, r_max=16), 0, "sgmv_stream_kernel"),
    (dict(M=200, d_in=1024, d_outs=[512, 256, 256], n_pool=20, r_max=32), 0, "sgmv_small_kernel"),
    (dict(M=600, d_in=512, d_outs=[256, 128], n_pool=10, r_max=64, ranks=[8, 64], run_len=40), 0, None),
    (dict(M=5000, d_in=256, d_outs=[256, 128, 128], n_pool=60, r_max=16, run_len=50), 0, None),
]


@pytest.mark.parametrize("ci", range(len(PER_SLICE_A_CASES)))
def test_per_slice_a(B, ci):
    kw, path, kernel = PER_SLICE_A_CASES[ci]
    w = wl.random_batch(seed=980 + ci, dtype="bf16", **kw)
    rng = np.random.default_rng(981 + ci)
    A_pools = [w.A] + [wl.round_bf16((rng.standard_normal(w.A.shape) / np.sqrt(w.A.shape[2])).astype(np.float32))
                       for _ in w.B[1:]]
    d = to_dev(w)
    A_dev = [torch.from_numpy(a).to(device="cuda", dtype=torch.bfloat16) for a in A_pools]
    batch = B.lora_prepare_batch(d["ids"], w.n_adapters, w.chunk_size)
    y = d["y"].clone()
    B.lora_delta(batch, d["x"], A_dev, d["B"], y, scale=w.scale, adapter_scale=d["adapter_scale"],
                 ranks=d["ranks"], path=path)
    if kernel is not None:
        assert B.KERNEL_NAMES.get(B.lora_last_kernels()) == kernel
    torch.cuda.synchronize()
    yg = y.float().cpu().numpy().astype(np.float64)
    ref = oracle.delta(w.x, w.ids, A_pools, w.B, w.y, scale=w.scale, adapter_scale=w.adapter_scale,
                       ranks=w.ranks)
    act = active_rows(w)
    assert rel_err(yg, ref, w.y.astype(np.float64), act) <= TOL["bf16"]
    assert np.array_equal(yg[~act], w.y[~act].astype(np.float64))
    assert batch.counts()["device_error"] == 0


# ----------------------------------------- rank-major B pools [n][r][d_out]

# per-slice A pools with rank-major B: the stacked shrink, in one launch and
# (above 2048 rows) over consecutive row ranges
@pytest.mark.parametrize("M", [1000, 4200])
def test_per_slice_a_rank_major(B, M):
    w = wl.random_batch(seed=986 + M, dtype="bf16", M=M, d_in=512, d_outs=[512, 128, 128], n_pool=24, r_max=16,
                        ranks=[8, 16], run_len=30, skip_frac=0.05, per_adapter_scale=True)
    rng = np.random.default_rng(987)
    A_pools = [w.A] + [wl.round_bf16((rng.standard_normal(w.A.shape) / np.sqrt(w.A.shape[2])).astype(np.float32))
                       for _ in w.B[1:]]
    d = to_dev(w)
    A_dev = [torch.from_numpy(a).to(device="cuda", dtype=torch.bfloat16) for a in A_pools]
    Bt = [b.transpose(1, 2).contiguous() for b in d["B"]]  # (n, r_max, d_out)
    batch = B.lora_prepare_batch(d["ids"], w.n_adapters, 0)
    y = d["y"].clone()
    B.lora_delta(batch, d["x"], A_dev, Bt, y, scale=w.scale, adapter_scale=d["adapter_scale"],
                 ranks=d["ranks"], b_rank_major=True)
    assert B.lora_last_kernels() == B.KERNEL_STREAM
    torch.cuda.synchronize()
    yg = y.float().cpu().numpy().astype(np.float64)
    ref = oracle.delta(w.x, w.ids, A_pools, w.B, w.y, scale=w.scale, adapter_scale=w.adapter_scale,
                       ranks=w.ranks)
    act = active_rows(w)
    assert rel_err(yg, ref, w.y.astype(np.float64), act) <= TOL["bf16"]
    assert np.array_equal(yg[~act], w.y[~act].astype(np.float64))
    assert batch.counts()["device_error"] == 0


RANK_MAJOR_CASES = [
    dict(M=512, d_in=4096, d_outs=[14336], n_pool=100, r_max=64, ranks=[8, 16, 32, 64], skip_frac=0.25,
         per_adapter_scale=True),
    dict(M=300, d_in=1024, d_outs=[1024, 256, 256], n_pool=30, r_max=32, ranks=[8, 24, 32], run_len=12),
    dict(M=100, d_in=512, d_outs=[520], n_pool=8, r_max=16, ranks=[3, 16]),
    # above the streaming kernel's 2048 rows: consecutive launches over row ranges
    dict(M=4500, d_in=1024, d_outs=[2048], n_pool=40, r_max=32, ranks=[8, 16, 32], skip_frac=0.1,
         per_adapter_scale=True),
    dict(M=4096, d_in=512, d_outs=[768, 256], n_pool=16, r_max=16, ranks=[8, 16], run_len=64),
    dict(M=2049, d_in=256, d_outs=[512], n_pool=6, r_max=64, ranks=[16, 64], run_len=700),
]


@pytest.mark.parametrize("ci", range(len(RANK_MAJOR_CASES)))
def test_rank_major_b(B, ci):
    w = wl.random_batch(seed=990 + ci, dtype="bf16", pad_value=float("nan"), **RANK_MAJOR_CASES[ci])
    d = to_dev(w)
    Bt = [b.transpose(1, 2).contiguous() for b in d["B"]]  # (n, r_max, d_out)
    batch = B.lora_prepare_batch(d["ids"], w.n_adapters, 0)
    y = d["y"].clone()
    B.lora_delta(batch, d["x"], d["A"], Bt, y, scale=w.scale, adapter_scale=d["adapter_scale"],
                 ranks=d["ranks"], b_rank_major=True)
    assert B.lora_last_kernels() == B.KERNEL_STREAM
    torch.cuda.synchronize()
    _assert_delta(w, y.float().cpu().numpy().astype(np.float64))


def test_rank_major_b_unsupported_elsewhere(B):
    # the streaming kernel computes bf16 only
    w = wl.random_batch(seed=995, M=3000, d_in=256, d_outs=[128], n_pool=8, r_max=16, dtype="f32")
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], w.n_adapters, 0)
    with pytest.raises(B.LoraError) as e:
        B.lora_delta(batch, d["x"], d["A"], [b.transpose(1, 2).contiguous() for b in d["B"]], d["y"],
                     b_rank_major=True)
    assert e.value.status == B.LORA_ERR_UNSUPPORTED
