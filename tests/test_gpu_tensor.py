"""GPU parity of the tensor-core (tcgen05) path against the CPU oracle,
forced (PATH_TENSOR) and through the automatic split by segment length."""
import numpy as np
import pytest
import torch

from segmented_gather_gemv_gb300 import workloads as wl
from tests._lora_case import TOL, active_rows, oracle_delta, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from segmented_gather_gemv_gb300 import binding
    binding.lib()
    return binding


def _run(B, w, path, tc_min=0):
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], w.n_adapters, w.chunk_size, tc_min_rows=tc_min)
    y = d["y"]
    B.lora_delta(batch, d["x"], d["A"], d["B"], y, scale=w.scale, adapter_scale=d["adapter_scale"],
                 ranks=d["ranks"], path=path)
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64), batch


def _check(w, y):
    y_ref = oracle_delta(w)
    act = active_rows(w)
    err = rel_err(y, y_ref, w.y.astype(np.float64), act)
    assert err <= TOL[w.dtype], "rel err %.3e" % err
    assert np.array_equal(y[~act], w.y[~act].astype(np.float64)), "inactive rows changed"
    assert np.isfinite(y).all()
    return err


TC_CASES = [
    dict(M=128, d_in=256, d_outs=[128], n_pool=1, r_max=16, run_len=128),        # one full tile
    dict(M=200, d_in=512, d_outs=[384], n_pool=3, r_max=16, run_len=50),         # several segments
    dict(M=300, d_in=1000, d_outs=[776], n_pool=4, r_max=32, run_len=100),       # ragged d_in / d_out
    dict(M=333, d_in=4096, d_outs=[4096], n_pool=6, r_max=16, run_len=111),      # decode-like widths
    dict(M=257, d_in=520, d_outs=[264, 64, 136], n_pool=5, r_max=32, run_len=40,
         ranks=[8, 16, 24, 32], per_adapter_scale=True),                         # slices, mixed ranks
    dict(M=180, d_in=192, d_outs=[256], n_pool=7, r_max=24, run_len=3),          # scattered rows
    dict(M=64, d_in=128, d_outs=[128], n_pool=2, r_max=8, run_len=64),
    dict(M=400, d_in=328, d_outs=[200, 72], n_pool=3, r_max=16, run_len=77),     # 32-row groups + partial group, ragged slices
    dict(M=1100, d_in=4096, d_outs=[1024], n_pool=2, r_max=16, run_len=550),     # long contiguous runs
]


@pytest.mark.parametrize("ci", range(len(TC_CASES)))
def test_tensor_path_forced(B, ci):
    w = wl.random_batch(seed=400 + ci, dtype="bf16", **TC_CASES[ci])
    y, batch = _run(B, w, path=B.PATH_TENSOR)
    _check(w, y)
    assert batch.counts()["device_error"] == 0


@pytest.mark.parametrize("chunk", [0, 64, 48])
def test_tensor_path_chunks_merge(B, chunk):
    w = wl.random_batch(seed=420, M=700, d_in=384, d_outs=[512], n_pool=5, r_max=16,
                        run_len=175, dtype="bf16", chunk_size=chunk)
    y, _ = _run(B, w, path=B.PATH_TENSOR)
    _check(w, y)


def test_tensor_path_nan_padding(B):
    w = wl.random_batch(seed=430, M=256, d_in=512, d_outs=[384], n_pool=8, r_max=32,
                        ranks=[8, 16, 24, 32], run_len=32, dtype="bf16", pad_value=float("nan"),
                        per_adapter_scale=True)
    y, _ = _run(B, w, path=B.PATH_TENSOR)
    _check(w, y)


def test_tensor_path_rank_too_large_flags(B):
    w = wl.random_batch(seed=431, M=128, d_in=256, d_outs=[128], n_pool=2, r_max=128,
                        run_len=64, dtype="bf16", ranks=np.array([128, 64], np.int32))
    y, batch = _run(B, w, path=B.PATH_TENSOR)
    assert batch.counts()["device_error"] & B.DEVERR_RANK


@pytest.mark.parametrize("tc_min", [1, 16, 40])
def test_auto_split_mixed_lengths(B, tc_min):
    # prefill-like runs and decode-like single rows in one batch
    w = wl.mixed_serving(n_prefill_seq=3, prefill_rows=600, len_lo=64, len_hi=400, n_decode=90,
                         n_pool=16, r=32, d_in=1024, d_outs=(512, 256, 256))
    y, batch = _run(B, w, path=B.PATH_AUTO, tc_min=tc_min)
    _check(w, y)
    c = batch.counts()
    assert c["num_tc_segs"] + c["num_small_segs"] == c["num_segs"]


def test_auto_split_odd_rank_goes_to_cuda_cores(B):
    w = wl.random_batch(seed=440, M=300, d_in=256, d_outs=[256], n_pool=4, r_max=16, run_len=100,
                        ranks=np.array([12, 16, 4, 8], np.int32), dtype="bf16")
    y, batch = _run(B, w, path=B.PATH_AUTO, tc_min=16)
    _check(w, y)
    assert batch.counts()["device_error"] == 0


def test_tensor_and_cuda_core_paths_agree(B):
    w = wl.prefill(n_seq=4, len_lo=100, len_hi=300, d_in=1024, d_out=2048)
    y_tc, _ = _run(B, w, path=B.PATH_TENSOR)
    y_cc, _ = _run(B, w, path=B.PATH_CUDA_CORE)
    base = w.y.astype(np.float64)
    assert rel_err(y_tc, y_cc, base) <= 1e-2
    _check(w, y_tc)


def test_auto_split_rank64_long_segments_use_cuda_cores(B):
    w = wl.random_batch(seed=441, M=400, d_in=512, d_outs=[256], n_pool=4, r_max=64, run_len=100,
                        ranks=np.array([64, 16, 64, 32], np.int32), dtype="bf16", pad_value=float("nan"))
    y, batch = _run(B, w, path=B.PATH_AUTO, tc_min=16)
    _check(w, y)
    assert batch.counts()["device_error"] == 0


@pytest.mark.parametrize("n_decode", [0, 60, 106])
def test_auto_split_small_batch_both_kernels(B, n_decode):
    # the CUDA-core kernel starts first; here the tensor-core kernel after it
    # has long segments to do as well
    w = wl.mixed_serving(n_prefill_seq=2, prefill_rows=150, len_lo=64, len_hi=100, n_decode=n_decode,
                         n_pool=16, r=16, d_in=1024, d_outs=(512, 256, 256))
    assert w.M <= 256
    y, batch = _run(B, w, path=B.PATH_AUTO)
    _check(w, y)
    c = batch.counts()
    assert c["tc_rows"] > 0 and c["device_error"] == 0
    assert (c["num_small_segs"] > 0) == (n_decode > 0)


@pytest.mark.parametrize("M", [200, 256, 257, 600])
def test_auto_split_back_to_back_calls(B, M):
    # two calls in a row on one batch and one y (the second kernel pair starts
    # while the first may still be finishing): y gains the delta twice
    n_dec = M // 3
    w = wl.mixed_serving(n_prefill_seq=2, prefill_rows=M - n_dec, len_lo=64, len_hi=400, n_decode=n_dec,
                         n_pool=16, r=16, d_in=1024, d_outs=(512, 256, 256))
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], w.n_adapters, w.chunk_size)
    y = d["y"]
    for _ in range(2):
        B.lora_delta(batch, d["x"], d["A"], d["B"], y, scale=w.scale, path=B.PATH_AUTO)
    torch.cuda.synchronize()
    yg = y.float().cpu().numpy().astype(np.float64)
    base = w.y.astype(np.float64)
    once = oracle_delta(w)
    act = active_rows(w)
    assert rel_err(yg, base + 2.0 * (once - base), base, act) <= 2 * TOL[w.dtype]
    assert np.array_equal(yg[~act], base[~act])
    assert batch.counts()["tc_rows"] > 0


# ------------------------------- split calls (lora_shrink / lora_expand)

def _shrink_expand(B, w, path, tc_min=0, seed=0):
    """lora_shrink into a guarded h, then lora_expand of a seeded h (not the
    GPU's); both against the oracle's shrink and expand."""
    import oracle
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], w.n_adapters, w.chunk_size, tc_min_rows=tc_min)
    act = active_rows(w)
    guard = torch.full((w.M, w.r_max + 4), -777.0, device="cuda")
    h = guard[:, :w.r_max]
    B.lora_shrink(batch, d["x"], d["A"], h=h, ranks=d["ranks"], path=path)
    torch.cuda.synchronize()
    kernels = B.lora_last_kernels()
    assert torch.all(guard[:, w.r_max:] == -777.0), "h written past r_max"
    hg = h.cpu().numpy().astype(np.float64)
    assert np.all(hg[~act] == -777.0), "h rows outside segments written"
    h_ref = oracle.shrink(w.x, w.ids, w.A, ranks=w.ranks)
    err = np.abs(hg[act] - h_ref[act]).max() / np.abs(h_ref[act]).max()
    assert err <= TOL[w.dtype], "shrink rel err %.3e" % err
    rng = np.random.default_rng(seed)
    h_in = rng.standard_normal((w.M, w.r_max)).astype(np.float32)
    y = d["y"].clone()
    B.lora_expand(batch, torch.from_numpy(h_in).cuda(), d["B"], y, scale=w.scale,
                  adapter_scale=d["adapter_scale"], ranks=d["ranks"], path=path)
    torch.cuda.synchronize()
    y_ref = oracle.expand(h_in, w.ids, w.B, w.y, scale=w.scale, adapter_scale=w.adapter_scale, ranks=w.ranks)
    yg = y.float().cpu().numpy().astype(np.float64)
    e2 = rel_err(yg, y_ref, w.y.astype(np.float64), act)
    assert e2 <= TOL[w.dtype], "expand rel err %.3e" % e2
    assert np.array_equal(yg[~act], w.y[~act].astype(np.float64)), "inactive rows changed"
    assert batch.counts()["device_error"] == 0
    return kernels, B.lora_last_kernels()


@pytest.mark.parametrize("ci", range(len(TC_CASES)))
def test_tensor_shrink_expand_forced(B, ci):
    w = wl.random_batch(seed=450 + ci, dtype="bf16", **TC_CASES[ci])
    k_s, k_e = _shrink_expand(B, w, B.PATH_TENSOR, seed=451 + ci)
    assert k_s == B.KERNEL_TENSOR and k_e == B.KERNEL_TENSOR


@pytest.mark.parametrize("n_decode", [0, 60])
def test_shrink_expand_auto_split(B, n_decode):
    # long groups on the tensor-core kernel, the rest on the small-segment kernel
    w = wl.mixed_serving(n_prefill_seq=3, prefill_rows=2600, len_lo=300, len_hi=1200, n_decode=n_decode,
                         n_pool=16, r=16, d_in=1024, d_outs=(512, 256, 256))
    k_s, k_e = _shrink_expand(B, w, B.PATH_AUTO, seed=470 + n_decode)
    assert k_s & B.KERNEL_TENSOR and k_e & B.KERNEL_TENSOR


def test_tensor_shrink_rank_zero_rows(B):
    # with every segment forced onto the tensor-core kernel, rows of rank-0
    # adapters get zero h (they are in segments); mixed with rank-16 groups
    w = wl.random_batch(seed=480, M=300, d_in=512, d_outs=[256], n_pool=4, r_max=16, run_len=60,
                        ranks=[0, 16], dtype="bf16")
    _shrink_expand(B, w, B.PATH_TENSOR, seed=481)
