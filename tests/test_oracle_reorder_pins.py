"""Pins for the oracle's Morton reorder and sink blocks (Piecewise-Taylor-
Attention README: "Morton tile reorder + fused gather kernel", the knob
n_sink_blocks; routing of "PISA: Piecewise Sparse Attention Is Wiser for
Efficient Diffusion Transformers", Algorithm 1 step 2)."""

import itertools

import numpy as np
import pytest

from oracle import morton_permutation, reorder_heads, restore_heads, route, route_gaps


def test_morton_4x4_hand_worked():
    """1 x 4 x 4 grid: y bits at positions 1 and 4, x bits at 0 and 3, so the
    order walks the 2 x 2 quadrants in Z order, each quadrant in Z order:
    raster 0 1 4 5 | 2 3 6 7 | 8 9 12 13 | 10 11 14 15."""
    assert morton_permutation((1, 4, 4)).tolist() == [0, 1, 4, 5, 2, 3, 6, 7,
                                                       8, 9, 12, 13, 10, 11, 14, 15]


def test_morton_2x2x2_puts_t_first():
    """In a 2 x 2 x 2 cube the code is 4t + 2y + x, the raster index itself;
    a 2 x 1 x 2 grid (no y bit used) orders (t, x) as 4t + x: raster order."""
    assert morton_permutation((2, 2, 2)).tolist() == list(range(8))
    assert morton_permutation((2, 1, 2)).tolist() == [0, 1, 2, 3]
    # 1 x 2 x 2 with a 3-token prefix: prefix first, then y before x
    assert morton_permutation((1, 2, 2), n_prefix=3).tolist() == [0, 1, 2, 3, 4, 5, 6]


def _recursive_order(T, Y, X):
    """Independent definition: split the power-of-two box into 8 octants in
    (t, y, x) binary order and visit them recursively, keeping grid tokens."""
    side = 1
    while side < max(T, Y, X, 2):
        side *= 2
    out = []

    def visit(t0, y0, x0, s):
        if t0 >= T or y0 >= Y or x0 >= X:
            return
        if s == 1:
            out.append((t0 * Y + y0) * X + x0)
            return
        h = s // 2
        for dt, dy, dx in itertools.product((0, 1), repeat=3):
            visit(t0 + dt * h, y0 + dy * h, x0 + dx * h, h)

    visit(0, 0, 0, side)
    return out


@pytest.mark.parametrize("grid,prefix", [((3, 5, 7), 0), ((4, 4, 4), 0), ((2, 6, 3), 5),
                                         ((1, 9, 13), 2), ((5, 1, 1), 0)])
def test_morton_equals_recursive_octants(grid, prefix):
    perm = morton_permutation(grid, n_prefix=prefix)
    expect = list(range(prefix)) + [prefix + r for r in _recursive_order(*grid)]
    assert perm.tolist() == expect
    assert sorted(perm.tolist()) == list(range(prefix + int(np.prod(grid))))


def test_morton_blocks_of_eight_are_cubes():
    """In an 8 x 8 x 8 grid every 8 consecutive tokens form a 2 x 2 x 2 cube."""
    perm = morton_permutation((8, 8, 8))
    t, y, x = perm // 64, (perm // 8) % 8, perm % 8
    for b in range(64):
        s = slice(8 * b, 8 * b + 8)
        for c in (t[s], y[s], x[s]):
            assert c.max() - c.min() == 1 and c.min() % 2 == 0


def test_reorder_and_restore_are_inverse_transposes():
    rng = np.random.default_rng(0)
    N, H, D = 70, 3, 5
    perm = rng.permutation(N)
    x = rng.standard_normal((N, H, D))
    o = reorder_heads(x, perm)
    assert o.shape == (H, N, D)
    for h in range(H):
        for p in range(N):
            assert np.array_equal(o[h, p], x[perm[p], h])
    assert np.array_equal(restore_heads(o, perm), x)
    tok = np.broadcast_to(np.arange(N, dtype=np.float64)[:, None, None], (N, H, D))
    assert np.array_equal(reorder_heads(tok, perm)[1, :, 0], perm.astype(np.float64))


def _brute_sets(r, topk, band, n_sink):
    nb = r.shape[0]
    out = []
    for i in range(nb):
        forced = [j for j in range(nb) if abs(i - j) <= band or j < n_sink]
        cand = [j for j in range(nb) if j not in forced]
        kk = min(topk, len(cand))
        best_key, best = None, None
        for sub in itertools.combinations(cand, kk):
            key = (-sum(r[i, j] for j in sub), sub)
            if best_key is None or key < best_key:
                best_key, best = key, sub
        out.append(sorted(forced + list(best)))
    return out


@pytest.mark.parametrize("nb,topk,band,n_sink,seed", [(8, 2, 1, 1, 0), (9, 3, 0, 2, 1),
                                                       (7, 2, 1, 3, 2), (6, 4, 1, 6, 3)])
def test_sink_route_matches_brute_force(nb, topk, band, n_sink, seed):
    rng = np.random.default_rng(seed)
    qbar = rng.integers(-2, 3, size=(nb, 2)).astype(np.float64)
    kbar = rng.integers(-2, 3, size=(nb, 2)).astype(np.float64)
    sets = route(qbar, kbar, 1.0, topk, band, n_sink=n_sink)
    assert [list(s) for s in sets] == _brute_sets(qbar @ kbar.T, topk, band, n_sink)


def test_zero_sinks_is_the_plain_route_and_all_sinks_select_everything():
    rng = np.random.default_rng(7)
    nb = 20
    qbar, kbar = rng.standard_normal((nb, 4)), rng.standard_normal((nb, 4))
    a, b = route(qbar, kbar, 0.5, 3, 1), route(qbar, kbar, 0.5, 3, 1, n_sink=0)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    full = route(qbar, kbar, 0.5, 0, 0, n_sink=nb)
    assert all(s.tolist() == list(range(nb)) for s in full)
    g = route_gaps(qbar, kbar, 0.5, 3, 1, n_sink=4)
    assert np.all(np.isfinite(g[4:]))


def test_route_on_sampled_rows_equals_the_full_route():
    rng = np.random.default_rng(12)
    nb = 40
    qbar, kbar = rng.standard_normal((nb, 6)), rng.standard_normal((nb, 6))
    bias, bonus = rng.standard_normal(nb), rng.random((nb, nb))
    full = route(qbar, kbar, 0.4, 5, 1, bias=bias, n_sink=2, bonus=bonus)
    gfull = route_gaps(qbar, kbar, 0.4, 5, 1, bias=bias, n_sink=2, bonus=bonus)
    rows = [39, 0, 17, 3]
    part = route(qbar, kbar, 0.4, 5, 1, bias=bias, n_sink=2, bonus=bonus, rows=rows)
    gpart = route_gaps(qbar, kbar, 0.4, 5, 1, bias=bias, n_sink=2, bonus=bonus, rows=rows)
    for a, i in enumerate(rows):
        assert np.array_equal(part[a], full[i])
        assert gpart[a] == gfull[i]
