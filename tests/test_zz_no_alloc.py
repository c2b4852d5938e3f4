"""lora_prepare_batch_static (the library's own device workspace, no
allocation) against lora_prepare_batch with a caller workspace, through the
C ABI, on two calls in a row: metadata bit-exact, and the delta computed from
each batch within the bf16 tolerance.  The second call is smaller than the
first, so values a call leaves in the shared array must not leak into the
next batch.  Collected last on purpose; it also passes alone."""
import numpy as np
import pytest
import torch

from segmented_gather_gemv_gb300 import workloads as wl
from tests._lora_case import TOL, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from segmented_gather_gemv_gb300 import binding
    binding.lib()
    return binding


def _compare_batches(a, b):
    ga, gb = a.arrays(), b.arrays()
    S = ga["num_segs"]
    assert S == gb["num_segs"]
    for k in ("num_segs", "num_active", "num_invalid", "num_small_segs", "num_tc_segs", "tc_rows",
              "device_error", "num_groups"):
        assert ga[k] == gb[k], k
    for k in ("sorted_token_ids", "seg_indptr", "seg_lens", "weight_indices", "small_segs", "tc_segs", "tc_indptr"):
        assert torch.equal(ga[k], gb[k]), k
    ra, rb = ga["seg_records"], gb["seg_records"]
    assert torch.equal(ra[:S, :4], rb[:S, :4])  # {start, len, adapter, s}
    for s_ in range(S):  # inline rows: the first min(len, 28) are defined
        k = min(int(ra[s_, 1]), 28)
        assert torch.equal(ra[s_, 4:4 + k], rb[s_, 4:4 + k])
    assert (rb[S:, 1] == 0).all()  # descriptors past the last segment have len 0


def _delta(B, w, d, batch):
    y = d["y"].clone()
    B.lora_delta(batch, d["x"], d["A"], d["B"], y, scale=w.scale, adapter_scale=d["adapter_scale"],
                 ranks=d["ranks"])
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64)


CALLS = [
    dict(seed=900, M=700, d_in=512, d_outs=[384], n_pool=40, r_max=16, run_len=5, skip_frac=0.1, chunk_size=8),
    dict(seed=901, M=150, d_in=512, d_outs=[384], n_pool=40, r_max=16, run_len=3, skip_frac=0.1, chunk_size=8),
]


def test_static_workspace_prepare_matches_two_calls(B):
    for kw in CALLS:
        w = wl.random_batch(dtype="bf16", **kw)
        d = to_dev(w)
        ref = B.lora_prepare_batch(d["ids"], w.n_adapters, w.chunk_size)
        got = B.lora_prepare_batch_static(d["ids"], w.n_adapters, w.chunk_size)
        _compare_batches(ref, got)
        y_ref = _delta(B, w, d, ref)
        y_got = _delta(B, w, d, got)
        assert rel_err(y_got, y_ref, w.y.astype(np.float64)) <= TOL["bf16"]


def test_static_workspace_rejects_large_batch(B):
    M, n = 65536, 4096
    assert B.lora_workspace_size(M, n, 1) > 4 << 20
    ids = torch.zeros(M, dtype=torch.int32, device="cuda")
    with pytest.raises(B.LoraError) as e:
        B.lora_prepare_batch_static(ids, n, 1)
    assert e.value.status == B.LORA_ERR_WORKSPACE
