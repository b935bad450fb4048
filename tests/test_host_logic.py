"""Host-side logic of the Python binding that needs no GPU: head grouping of
the host pipeline, the density-to-top-k rule, the selected-list width, and
the one-call API's option checks (which run before any launch)."""

import pytest

from piecewise_sparse_attention_gb300 import pisa as P


@pytest.mark.parametrize("heads", [1, 2, 3, 5, 24, 40, 41, 136])
@pytest.mark.parametrize("chunks", [1, 2, 3, 4, 8, 10, 12, 64])
@pytest.mark.parametrize("taper", [False, True, 0.25])
def test_head_groups_partition_the_heads(heads, chunks, taper):
    b = P.head_groups(heads, chunks, taper)
    sizes = [b[i + 1] - b[i] for i in range(len(b) - 1)]
    assert b[0] == 0 and b[-1] == heads
    assert len(sizes) == min(chunks, heads)
    assert all(s >= 1 for s in sizes)
    if not taper or len(sizes) < 3:
        assert max(sizes) - min(sizes) <= 1
    elif heads >= 4 * len(sizes):
        # half-weight ends: the first and last groups are the smallest
        assert sizes[0] <= min(sizes[1:-1]) and sizes[-1] <= min(sizes[1:-1])


def test_taper_weight_must_be_a_fraction():
    for bad in (-0.5, 1.5):
        with pytest.raises(ValueError):
            P.head_groups(40, 10, bad)


def test_tapered_groups_of_the_bench_workload():
    assert P.head_groups(40, 10, True) == [0, 2, 7, 11, 16, 20, 24, 29, 33, 38, 40]
    assert P.head_groups(40, 8, False) == [0, 5, 10, 15, 20, 25, 30, 35, 40]


def test_topk_for_density_and_list_width():
    # k = ceil(density n_b): 11 of 72, 64 of 512, 128 of 1024 and of 2048 at 1/16
    assert P.topk_for_density(0.15, 72) == 11
    assert P.topk_for_density(0.125, 512) == 64
    assert P.topk_for_density(0.125, 1024) == 128
    assert P.topk_for_density(0.0625, 2048) == 128
    assert P.max_sel(512, 64, 1) == 67
    assert P.max_sel(16, 100, 1) == 16
    assert P.max_sel(1, 0, 0) == 1


def test_bench_stats_and_route_roofline_arithmetic():
    """The bench line's stats and route roofline objects: algorithmic bytes and
    score FMAs from the shapes alone, fractions against the stated peaks."""
    import bench

    H, n, d = 40, 32760, 128
    nb = -(-n // 64)
    st = bench.stats_roofline(H, n, d, nb, 0.1)
    # Q and K read once in bf16, qbar and kbar written in float32
    assert st["bytes_per_launch"] == 2 * H * n * d * 2 + 2 * H * nb * d * 4 == 691896320
    assert st["achieved"] == pytest.approx(691896320 / 1e-4 / 1e9)
    assert st["frac"] == pytest.approx(st["achieved"] / st["peak"])
    assert st["bound"] == "hbm" and st["unit"] == "GB/s"
    ms = 67
    rt = bench.route_roofline(H, nb, d, ms, 0.5, {"sm_mhz": 2000.0})
    assert rt["bytes_per_launch"] == 2 * H * nb * d * 4 + H * nb * (ms + 1) * 4
    # one f32 FMA per channel per (query block, key block) pair
    assert rt["achieved_tfma"] == pytest.approx(H * nb * nb * d / 5e-4 / 1e12)
    assert rt["peak_tfma"] == pytest.approx(152 * 128 * 2000e6 / 1e12)
    assert rt["frac"] == pytest.approx(rt["achieved_tfma"] / rt["peak_tfma"])
    # no clock samples: the maximum SM clock stands in
    assert bench.route_roofline(H, nb, d, ms, 0.5, None)["peak_tfma"] == pytest.approx(
        152 * 128 * 2070e6 / 1e12)


def test_bench_sample_parity_counts_routes_and_compares_rows():
    """The bench line's parity figures: a route row that differs counts as a
    near-tie only where the stored gap is below 1e-5, and the output rows of a
    query block are compared only where its route agrees."""
    import types

    import numpy as np
    import torch

    import bench

    wl = types.SimpleNamespace(nb=3, block=2, band=0, topk=1)
    n, d = 6, 4
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((n, d))
    bench._ORACLE_SAMPLE.clear()
    bench._ORACLE_SAMPLE[0] = {
        "sets": [[0, 1], [1, 2], [0, 2]],
        "gaps": np.array([0.1, 1e-7, 0.5]),
        "out": {0: ref[0:2], 2: ref[4:6]},
        # row 1: blocks 0 and 2 tie within 1e-7, so either is a valid pick
        "scores": np.array([[0.0, 0.2, 0.1], [0.3, 0.0, 0.3 - 1e-7], [0.9, 0.4, 0.0]]),
    }
    # row 1 differs at a near-tie, row 2 differs with a large gap (a failure)
    idx = torch.tensor([[[0, 1], [0, 1], [1, 2]]], dtype=torch.int32)
    cnt = torch.tensor([[2, 2, 2]], dtype=torch.int32)
    got = ref + 1e-3
    fwd32 = torch.from_numpy(got[None]).float()
    out16 = torch.from_numpy(got[None]).to(torch.bfloat16)
    try:
        r = bench.sample_parity(wl, idx, cnt, fwd32, out16)
    finally:
        bench._ORACLE_SAMPLE.clear()
    assert r["route_rows"] == 3 and r["route_rows_identical"] == 1
    assert r["route_rows_near_tie"] == 1 and r["route_rows_failing"] == 1
    assert r["query_blocks_compared"] == 1  # block 2's route is wrong: not compared
    assert abs(r["max_abs_f32_out"] - 1e-3) < 1e-6
    assert r["min_row_cosine_f32_out"] > 0.9999
    assert r["pass"] is False


def test_bench_near_tie_rows_must_be_valid_selections():
    """A differing row at a near-tie passes only as a valid top-k: the band
    block present, the right count, no repeats, scores within 1e-5 of the
    boundary."""
    import types

    import numpy as np

    import bench

    wl = types.SimpleNamespace(nb=4, band=0, topk=1)
    r = np.array([0.5, 0.0, 0.5 - 1e-7, 0.1])  # query block 1: blocks 0 and 2 tie
    assert bench.valid_near_tie([0, 1], r, 1, wl)
    assert bench.valid_near_tie([1, 2], r, 1, wl)
    assert not bench.valid_near_tie([1, 3], r, 1, wl)      # below the tie
    assert not bench.valid_near_tie([0, 2], r, 1, wl)      # band block 1 dropped
    assert not bench.valid_near_tie([0, 1, 2], r, 1, wl)   # one too many
    assert not bench.valid_near_tie([2, 1], r, 1, wl)      # not ascending


def test_bench_hybrid_flops_follow_the_plan():
    """The bench counts the hybrid kernel's executed tensor FLOPs under the plan
    the call used: per 128-row query tile, ceil(|union of its two blocks'
    critical sets| / 2) exact tiles, plus the hi/lo centroid tiles and the Q
    Hbar products of every tile slot (an empty slot still runs those)."""
    import bench
    import torch

    H, nb, ms = 2, 5, 4
    # critical sets of the 5 query blocks of each head (padding entries past
    # cnt, and out-of-range entries, are ignored)
    idx = torch.tensor([[[0, 1, 2, 9], [1, 2, 3, 0], [2, 3, 4, 0], [3, 4, 0, 0], [4, 0, 0, 0]],
                        [[0, 0, 0, 0], [1, 4, 0, 0], [2, 7, 0, 0], [3, 1, 0, 0], [4, 1, 2, 3]]],
                       dtype=torch.int32)
    cnt = torch.tensor([[3, 3, 3, 2, 1], [1, 2, 2, 2, 4]], dtype=torch.int32)
    # 2 CTAs per head = 4 tile slots; head 0 pairs neighbours, head 1 matches
    # blocks 1 + 4 and 0 + 2, then 3 alone, then an empty slot
    plan = torch.tensor([[[0, 1, 2, 3], [4, 5, 5, 5]],
                         [[1, 4, 0, 2], [3, 5, 5, 5]]], dtype=torch.int32)
    unions = [4, 3, 1, 0] + [4, 2, 2, 0]  # |S_a | S_b| per slot, in plan order
    exact = sum((u + 1) // 2 for u in unions)
    mm = 2.0 * 128 ** 3
    slots = H * 4
    want = exact * 2 * mm + slots * 1 * 2 * (2 * mm) + slots * 2 * mm
    assert bench.hybrid_forward_flops(idx, cnt, nb, H, plan, torch) == want

    # the plan sits after the operand copies, at the next 256-byte boundary
    d, n = 64, 5 * 64 - 3
    off = -(-((4 * H * nb * d + 2 * H * d * d) * 2) // 256) * 256
    ws = torch.zeros(off + H * 4 * 2 * 4, dtype=torch.uint8)
    ws[off:].view(torch.int32).copy_(plan.reshape(-1))
    assert torch.equal(bench.hybrid_plan(ws, H, n, d, nb), plan)
    with pytest.raises(RuntimeError):
        bench.hybrid_plan(ws[:-4], H, n, d, nb)
