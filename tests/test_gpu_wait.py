"""The bounded device waits give up and report instead of hanging: a CTA
waits on a barrier that nothing completes (no copy in flight), the wait runs
out, LORA_DEVERR_WAIT is set in the counters, and the context stays usable."""
import numpy as np
import pytest
import torch

from segmented_gather_gemv_gb300 import workloads as wl
from tests._lora_case import TOL, active_rows, oracle_delta, rel_err, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_and_returns():
    from segmented_gather_gemv_gb300 import binding as B
    counts = torch.zeros(len(B.COUNT_NAMES), dtype=torch.int32, device="cuda")
    B.lora_selftest_wait(counts)
    torch.cuda.synchronize()
    c = counts.cpu().numpy()
    assert c[B.COUNT_NAMES.index("device_error")] & B.DEVERR_WAIT
    assert (np.delete(c, B.COUNT_NAMES.index("device_error")) == 0).all()
    # the context still runs the path afterwards
    w = wl.random_batch(seed=11, M=64, d_in=256, d_outs=[128], n_pool=4, r_max=16, dtype="bf16")
    d = to_dev(w)
    batch = B.lora_prepare_batch(d["ids"], w.n_adapters, 0)
    B.lora_delta(batch, d["x"], d["A"], d["B"], d["y"], scale=w.scale)
    torch.cuda.synchronize()
    got = d["y"].float().cpu().numpy().astype(np.float64)
    assert rel_err(got, oracle_delta(w), w.y.astype(np.float64), active_rows(w)) <= TOL["bf16"]
    assert batch.counts()["device_error"] == 0
