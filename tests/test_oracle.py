"""Pins for the CPU oracle: each test checks it against something other than
itself -- a worked example printed on the pages, a closed form, an invariant,
a special case that reduces to a library routine, or brute force on tiny
inputs.  No GPU needed."""
import json
import os

import numpy as np
import pytest

import oracle
from segmented_gather_gemv_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- grouping

def test_segment_example_from_punica_page():
    g = _golden("punica_segment_example.json")
    out = oracle.prepare_batch(g["ids"], g["n_adapters"], g["chunk_size"])
    assert out["seg_indptr"].tolist() == g["seg_indptr"]
    assert out["seg_lens"].tolist() == g["seg_lens"]
    assert out["weight_indices"].tolist() == g["weight_indices"]
    assert out["sorted_token_ids"].tolist() == g["sorted_token_ids"]
    assert out["num_segs"] == 3 and out["num_active"] == 7 and out["num_invalid"] == 0


def _brute_grouping(ids, n, chunk):
    """Independent statement of the grouping rule: stable sort of the valid
    rows by the position at which their adapter first occurs."""
    ids = list(ids)
    first = {}
    for i, a in enumerate(ids):
        if 0 <= a < n and a not in first:
            first[a] = i
    rows = sorted((i for i, a in enumerate(ids) if 0 <= a < n),
                  key=lambda i: (first[ids[i]], i))
    segs = []  # (start, len, adapter)
    p = 0
    while p < len(rows):
        a = ids[rows[p]]
        q = p
        while q < len(rows) and ids[rows[q]] == a:
            q += 1
        if chunk > 0:
            for c in range(p, q, chunk):
                segs.append((c, min(chunk, q - c), a))
        else:
            segs.append((p, q - p, a))
        p = q
    return rows, segs


def test_page1_routing_grouping():
    g = _golden("page1_test_shape.json")
    out = oracle.prepare_batch(g["lora_indices"], g["num_loras"])
    rows, segs = _brute_grouping(g["lora_indices"], g["num_loras"], 0)
    assert out["sorted_token_ids"].tolist() == rows == [0, 3, 1, 2]
    assert out["seg_indptr"].tolist() == [0, 2, 3, 4]
    assert out["weight_indices"].tolist() == [2, 0, 1]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("chunk", [0, 1, 3, 64, 1000])
def test_grouping_brute_force(seed, chunk):
    rng = np.random.default_rng(seed)
    M = int(rng.integers(0, 300))
    n = int(rng.integers(1, 40))
    ids = rng.integers(-1, n + 3, size=M).astype(np.int32)  # -1, valid, out of range
    out = oracle.prepare_batch(ids, n, chunk)
    rows, segs = _brute_grouping(ids, n, chunk)
    assert out["sorted_token_ids"].tolist() == rows
    assert [(int(s), int(l), int(a)) for s, l, a in zip(out["seg_indptr"][:-1], out["seg_lens"], out["weight_indices"])] == segs
    assert out["num_invalid"] == int(((ids >= n) | (ids < -1)).sum())
    assert out["num_active"] == int(((ids >= 0) & (ids < n)).sum())
    # invariants
    ind = out["seg_indptr"]
    assert ind[0] == 0 and ind[-1] == out["num_active"]
    assert np.all(np.diff(ind) > 0)
    assert np.array_equal(np.diff(ind), out["seg_lens"])
    assert sorted(out["sorted_token_ids"].tolist()) == [i for i in range(M) if 0 <= ids[i] < n]
    for s in range(out["num_segs"]):
        seg_rows = out["sorted_token_ids"][ind[s]:ind[s + 1]]
        assert np.all(ids[seg_rows] == out["weight_indices"][s])
        assert np.all(np.diff(seg_rows) > 0)
        if chunk:
            assert out["seg_lens"][s] <= chunk


def test_ascending_order_punica_ids():
    # the "III.Punica" page's ids 2 2 2 5 5 1 1, grouped by increasing adapter
    # id instead of first appearance: adapter 1 (rows 5, 6), then 2, then 5
    out = oracle.prepare_batch([2, 2, 2, 5, 5, 1, 1], 6, ascending=True)
    assert out["sorted_token_ids"].tolist() == [5, 6, 0, 1, 2, 3, 4]
    assert out["seg_indptr"].tolist() == [0, 2, 5, 7]
    assert out["weight_indices"].tolist() == [1, 2, 5]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("chunk", [0, 1, 3, 64])
def test_ascending_order_is_a_stable_sort(seed, chunk):
    # ascending grouping = numpy's stable sort of the valid rows by id, each
    # group then cut into chunks
    rng = np.random.default_rng(100 + seed)
    M = int(rng.integers(0, 300))
    n = int(rng.integers(1, 40))
    ids = rng.integers(-1, n + 3, size=M).astype(np.int32)
    out = oracle.prepare_batch(ids, n, chunk, ascending=True)
    valid = np.nonzero((ids >= 0) & (ids < n))[0]
    rows = valid[np.argsort(ids[valid], kind="stable")]
    assert out["sorted_token_ids"].tolist() == rows.tolist()
    segs = []
    pos = 0
    for a in np.unique(ids[valid]):
        L = int((ids[valid] == a).sum())
        step = chunk if chunk else L
        for c in range(0, L, step):
            segs.append((pos + c, min(step, L - c), int(a)))
        pos += L
    assert [(int(s), int(l), int(a)) for s, l, a in zip(out["seg_indptr"][:-1], out["seg_lens"], out["weight_indices"])] == segs
    # the same segments as first-appearance order, only reordered
    fa = oracle.prepare_batch(ids, n, chunk)
    assert sorted(fa["weight_indices"].tolist()) == sorted(out["weight_indices"].tolist())
    assert out["num_segs"] == fa["num_segs"] and out["num_active"] == fa["num_active"]


def test_grouping_degenerate_cases():
    assert oracle.prepare_batch([], 5)["num_segs"] == 0
    out = oracle.prepare_batch([-1, -1, 9], 5)
    assert out["num_segs"] == 0 and out["num_active"] == 0 and out["num_invalid"] == 1
    out = oracle.prepare_batch([4, 4, 4, 4, 4], 5, chunk_size=2)
    assert out["seg_lens"].tolist() == [2, 2, 1]
    assert out["weight_indices"].tolist() == [4, 4, 4]


# ---------------------------------------------------------------- values

def _brute_delta(w: wl.Workload, scale_mult=1.0):
    """Per-adapter dense matmuls over the row subset of each adapter
    (numpy float64 matmul), independent of the oracle's per-token loop."""
    n = w.n_adapters
    x = w.x.astype(np.float64)
    y = w.y.astype(np.float64).copy()
    col = 0
    offs = []
    for d in w.d_outs:
        offs.append(col)
        col += d
    for a in range(n):
        rows = np.nonzero(w.ids == a)[0]
        if rows.size == 0:
            continue
        r = w.r_max if w.ranks is None else int(w.ranks[a])
        s = (w.scale if w.adapter_scale is None else float(w.adapter_scale[a])) * scale_mult
        Aa = w.A[a, :r, :].astype(np.float64)           # (r, d_in)
        H = x[rows] @ Aa.T                               # (rows, r)
        for B, off in zip(w.B, offs):
            Ba = B[a, :, :r].astype(np.float64)         # (d_out, r)
            y[np.ix_(rows, np.arange(off, off + B.shape[1]))] += s * (H @ Ba.T)
    return y


def _run_oracle(w: wl.Workload, scale=None, return_h=False):
    return oracle.delta(w.x, w.ids, w.A, w.B, w.y,
                        scale=w.scale if scale is None else scale,
                        adapter_scale=w.adapter_scale, ranks=w.ranks,
                        return_h=return_h)


def _rel_err(a, b, base):
    d = np.abs(a - b).max() if a.size else 0.0
    ref = np.abs(b - base).max() if b.size else 0.0
    return d / max(ref, 1e-300)


def test_page1_shape_brute_force_and_page_tolerance():
    g = _golden("page1_test_shape.json")
    w = wl.page1_toy()
    assert list(w.A.shape) == g["a_pool_shape"] and list(w.B[0].shape) == g["b_pool_shape"]
    assert w.ids.tolist() == g["lora_indices"]
    y = _run_oracle(w)
    ref = _brute_delta(w)
    assert _rel_err(y, ref, w.y) < 1e-13
    # The page's own check: its fp32 per-token loop agrees within 1e-3.
    page_loop = np.stack([(w.x[i][None] @ w.A[a].T) @ w.B[0][a].T
                          for i, a in enumerate(w.ids)])[:, 0, :]
    assert np.abs(page_loop.astype(np.float64) - y).max() < g["abs_tolerance"]


@pytest.mark.parametrize("case", [
    dict(M=37, d_in=48, d_outs=[40], n_pool=5, r_max=8),
    dict(M=50, d_in=24, d_outs=[16, 8, 24], n_pool=7, r_max=16, skip_frac=0.2, bad_frac=0.1),
    dict(M=64, d_in=32, d_outs=[56], n_pool=9, r_max=16, ranks=[4, 8, 16], per_adapter_scale=True),
    dict(M=33, d_in=40, d_outs=[24], n_pool=4, r_max=8, run_len=6, skip_frac=0.3),
])
def test_delta_brute_force(case):
    w = wl.random_batch(seed=3, dtype="f32", **case)
    y = _run_oracle(w)
    assert _rel_err(y, _brute_delta(w), w.y) < 1e-12


def test_single_adapter_reduces_to_matmul_chain():
    w = wl.random_batch(seed=5, M=21, d_in=30, d_outs=[26], n_pool=1, r_max=6, dtype="f32")
    y = _run_oracle(w)
    x, A, B = (v.astype(np.float64) for v in (w.x, w.A[0], w.B[0][0]))
    chain = w.y.astype(np.float64) + w.scale * np.linalg.multi_dot([x, A.T, B.T])
    assert _rel_err(y, chain, w.y) < 1e-12


def test_merged_weight_identity():
    """x W^T + s (x A^T) B^T == x (W + s B A)^T for one adapter
    ("vLLM-Ascend LoRA" article, sections 1.1 and 5.2; Punica page, SGMV:
    x@(W + A@B) == x@W + x@A@B)."""
    rng = np.random.default_rng(11)
    M, d_in, d_out, r, s = 19, 36, 28, 4, 0.75
    x = rng.standard_normal((M, d_in)).astype(np.float32)
    W = rng.standard_normal((d_out, d_in))
    A = rng.standard_normal((1, r, d_in)).astype(np.float32)
    B = rng.standard_normal((1, d_out, r)).astype(np.float32)
    ids = np.zeros(M, np.int32)
    base = x.astype(np.float64) @ W.T
    y = oracle.delta(x, ids, A, B, base, scale=s)
    merged = x.astype(np.float64) @ (W + s * B[0].astype(np.float64) @ A[0].astype(np.float64)).T
    assert np.abs(y - merged).max() / np.abs(merged).max() < 1e-12


def test_permutation_invariance_bit_exact():
    w = wl.random_batch(seed=8, M=45, d_in=32, d_outs=[24, 8], n_pool=6, r_max=8,
                        dtype="f32", skip_frac=0.2, ranks=[2, 4, 8])
    perm = np.random.default_rng(0).permutation(w.M)
    y = _run_oracle(w)
    yp = oracle.delta(w.x[perm], w.ids[perm], w.A, w.B, w.y[perm], scale=w.scale,
                      ranks=w.ranks)
    assert np.array_equal(yp, y[perm])


def test_scale_linearity_and_zero_scale():
    w = wl.random_batch(seed=9, M=30, d_in=16, d_outs=[20], n_pool=3, r_max=4,
                        dtype="f32", y_zero=True)
    d1 = _run_oracle(w, scale=0.375)
    d2 = _run_oracle(w, scale=0.75)
    assert np.array_equal(2.0 * d1, d2)     # power-of-two multiple: exact
    d3 = _run_oracle(w, scale=3 * 0.375)
    assert np.abs(d3 - 3 * d1).max() <= 1e-13 * np.abs(d3).max()
    w2 = wl.random_batch(seed=9, M=30, d_in=16, d_outs=[20], n_pool=3, r_max=4, dtype="f32")
    assert np.array_equal(_run_oracle(w2, scale=0.0), w2.y.astype(np.float64))


def test_skipped_and_invalid_rows_untouched():
    w = wl.random_batch(seed=12, M=40, d_in=16, d_outs=[12], n_pool=4, r_max=4,
                        dtype="f32", skip_frac=0.3, bad_frac=0.1)
    y = _run_oracle(w)
    idle = (w.ids < 0) | (w.ids >= w.n_adapters)
    assert idle.sum() > 0
    assert np.array_equal(y[idle], w.y[idle].astype(np.float64))
    assert not np.array_equal(y[~idle], w.y[~idle].astype(np.float64))


def test_mixed_rank_padding_is_never_read():
    """Rank mask ("vLLM-Ascend LoRA" article, section 3.4): NaN padding gives
    the same result as zero padding, and each adapter's result equals that
    of a pool sliced to its own rank."""
    kw = dict(seed=13, M=48, d_in=24, d_outs=[20, 12], n_pool=6, r_max=16,
              dtype="f32", ranks=[2, 4, 8, 16], per_adapter_scale=True)
    w0 = wl.random_batch(pad_value=0.0, **kw)
    wn = wl.random_batch(pad_value=float("nan"), **kw)
    y0, h0 = _run_oracle(w0, return_h=True)
    yn, hn = _run_oracle(wn, return_h=True)
    assert np.isfinite(yn).all()
    assert np.array_equal(y0, yn)
    act = w0.ids >= 0
    assert np.array_equal(h0[act], hn[act])
    for a in range(w0.n_adapters):
        rows = np.nonzero(w0.ids == a)[0]
        if rows.size == 0:
            continue
        r = int(w0.ranks[a])
        ys = oracle.delta(w0.x[rows], np.zeros(rows.size, np.int32), w0.A[a:a + 1, :r],
                          [B[a:a + 1, :, :r] for B in w0.B], w0.y[rows],
                          scale=float(w0.adapter_scale[a]))
        assert np.array_equal(ys, y0[rows])


def test_shrink_then_expand_equals_delta():
    w = wl.random_batch(seed=14, M=35, d_in=20, d_outs=[16, 4], n_pool=5, r_max=8,
                        dtype="f32", ranks=[3, 8], skip_frac=0.2, per_adapter_scale=True)
    h = oracle.shrink(w.x, w.ids, w.A, ranks=w.ranks)
    y2 = oracle.expand(h, w.ids, w.B, w.y, scale=w.scale,
                       adapter_scale=w.adapter_scale, ranks=w.ranks)
    y1, h1 = _run_oracle(w, return_h=True)
    act = (w.ids >= 0) & (w.ids < w.n_adapters)
    assert np.array_equal(h[act], h1[act])
    assert np.array_equal(y1, y2)
    # h is the unscaled intermediate: compare with a library matmul.
    for i in np.nonzero(act)[0]:
        a = w.ids[i]
        r = int(w.ranks[a])
        ref = w.A[a, :r].astype(np.float64) @ w.x[i].astype(np.float64)
        assert np.allclose(h[i, :r], ref, rtol=1e-13, atol=1e-13)
        assert np.all(h[i, r:] == 0)


def test_round_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    v = np.random.default_rng(1).standard_normal(10000).astype(np.float32) * 7
    v[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]  # ties
    ours = wl.round_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("case", range(3))
def test_parallel_delta_is_bit_identical(case):
    # the all-core variant shares the rows out over host threads; each row's
    # arithmetic is that of the serial loop, so the results must be identical
    kw = [dict(M=300, d_in=96, d_outs=[64, 32], n_pool=7, r_max=16, skip_frac=0.2, bad_frac=0.05),
          dict(M=129, d_in=64, d_outs=[40], n_pool=9, r_max=32, ranks=[8, 16, 24, 32],
               per_adapter_scale=True),
          dict(M=1, d_in=32, d_outs=[16], n_pool=2, r_max=8)][case]
    w = wl.random_batch(seed=900 + case, dtype="f32", **kw)
    y1 = oracle.delta(w.x, w.ids, w.A, w.B, w.y, scale=w.scale, adapter_scale=w.adapter_scale,
                      ranks=w.ranks)
    y4 = oracle.delta(w.x, w.ids, w.A, w.B, w.y, scale=w.scale, adapter_scale=w.adapter_scale,
                      ranks=w.ranks, threads=4)
    assert np.array_equal(y1, y4)
    assert oracle.delta.last_threads >= 1


# ---- per-slice A (a fused projection whose slices each have their own A)

def _brute_delta_per_slice_a(w, A_pools):
    x = w.x.astype(np.float64)
    y = w.y.astype(np.float64).copy()
    col = 0
    for A_t, B in zip(A_pools, w.B):
        for a in range(w.n_adapters):
            rows = np.nonzero(w.ids == a)[0]
            if rows.size == 0:
                continue
            r = w.r_max if w.ranks is None else int(w.ranks[a])
            s = w.scale if w.adapter_scale is None else float(w.adapter_scale[a])
            H = x[rows] @ A_t[a, :r, :].astype(np.float64).T
            y[np.ix_(rows, np.arange(col, col + B.shape[1]))] += s * (H @ B[a, :, :r].astype(np.float64).T)
        col += B.shape[1]
    return y


@pytest.mark.parametrize("case", [
    dict(M=40, d_in=32, d_outs=[24, 8, 16], n_pool=6, r_max=8, skip_frac=0.2),
    dict(M=29, d_in=48, d_outs=[16, 16], n_pool=4, r_max=16, ranks=[4, 8, 16], per_adapter_scale=True),
])
def test_per_slice_a_brute_force(case):
    w = wl.random_batch(seed=11, dtype="f32", **case)
    rng = np.random.default_rng(12)
    A_pools = [w.A] + [rng.standard_normal(w.A.shape).astype(np.float32) for _ in w.B[1:]]
    y = oracle.delta(w.x, w.ids, A_pools, w.B, w.y, scale=w.scale, adapter_scale=w.adapter_scale,
                     ranks=w.ranks)
    assert _rel_err(y, _brute_delta_per_slice_a(w, A_pools), w.y) < 1e-12
    # a slice's A pool changes only that slice's columns
    A2 = list(A_pools)
    A2[-1] = A2[-1] * 2
    y2 = oracle.delta(w.x, w.ids, A2, w.B, w.y, scale=w.scale, adapter_scale=w.adapter_scale,
                      ranks=w.ranks)
    last = sum(w.d_outs[:-1])
    assert np.array_equal(y2[:, :last], y[:, :last])
    act = (w.ids >= 0) & (w.ids < w.n_adapters)
    assert np.allclose(y2[act, last:] - w.y[act, last:], 2 * (y[act, last:] - w.y[act, last:]), rtol=1e-12, atol=1e-12)


def test_per_slice_a_equal_pools_is_the_shared_a():
    w = wl.random_batch(seed=13, M=33, d_in=40, d_outs=[24, 8], n_pool=5, r_max=8, dtype="f32",
                        skip_frac=0.1)
    shared = oracle.delta(w.x, w.ids, w.A, w.B, w.y, scale=w.scale)
    per = oracle.delta(w.x, w.ids, [w.A, w.A], w.B, w.y, scale=w.scale)
    assert np.array_equal(shared, per)
