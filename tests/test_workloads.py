"""The seeded input generator: determinism, exactness in the workload dtype,
shapes and the structure the workloads are meant to have."""

import numpy as np
import pytest

from piecewise_sparse_attention_gb300.workloads import (
    WORKLOADS, bf16_bits, make_head, make_inputs, round_to_bf16, small_case, token_coords)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e-8, 1e30], dtype=np.float32)
    r = round_to_bf16(x)
    import torch

    t = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(r, t)
    assert np.array_equal(round_to_bf16(r), r)


def test_generator_is_deterministic_and_per_head():
    wl = WORKLOADS["tiny"]
    a = make_inputs(wl)
    b = make_inputs(wl)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    q1, k1, v1 = make_head(wl, 1)
    assert np.array_equal(q1, a[0][1]) and np.array_equal(v1, a[2][1])
    assert not np.array_equal(a[0][0], a[0][1])


@pytest.mark.parametrize("name", ["flux", "wan"])
def test_bf16_workloads_are_exact_and_shaped(name):
    wl = WORKLOADS[name]
    q, k, v = make_head(wl, 0)
    for x in (q, k, v):
        assert x.shape == (wl.n, wl.d) and x.dtype == np.float32
        assert np.array_equal(round_to_bf16(x), x)
        assert np.isfinite(x).all()
    assert abs(v.std() - 1.0) < 0.02
    if wl.n_outliers:
        big = np.argsort(np.abs(q).mean(axis=0))[-wl.n_outliers:]
        bigk = np.argsort(np.abs(k).mean(axis=0))[-wl.n_outliers:]
        assert set(big) == set(bigk)


def test_workload_table():
    t = {n: (w.heads, w.n, w.d, w.nb, w.topk, w.band, w.dtype) for n, w in WORKLOADS.items()}
    assert t["tiny"] == (2, 1024, 64, 16, 4, 1, "f32")
    assert t["flux"] == (24, 4608, 128, 72, 11, 1, "bf16")
    assert t["wan"] == (40, 32760, 128, 512, 64, 1, "bf16")
    assert t["hunyuan"] == (24, 65536, 128, 1024, 128, 1, "bf16")
    assert t["long"] == (16, 131072, 128, 2048, 128, 1, "bf16")


def test_morton_order_is_a_permutation_with_compact_blocks():
    t, y, x = token_coords((21, 30, 52), "morton")
    n = 21 * 30 * 52
    assert len(set(zip(t.tolist(), y.tolist(), x.tolist()))) == n
    # a 64-token Morton block spans a compact neighbourhood
    spans = [max(np.ptp(c[i:i + 64]) for c in (t, y, x)) for i in range(0, n - 64, 64 * 37)]
    assert np.median(spans) <= 8
    tr, yr, xr = token_coords((4, 16, 16), "raster")
    assert list(xr[:3]) == [0, 1, 2] and tr[-1] == 3


def test_small_case_and_bits():
    q, k, v = small_case(2, 100, 8, seed=3)
    assert q.shape == (2, 100, 8)
    bits = bf16_bits(q)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, q)
