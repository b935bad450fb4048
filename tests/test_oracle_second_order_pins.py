"""Pins for the oracle's second-order block mass (Piecewise-Taylor-Attention
README, "Blog post": sum_n exp(q.k_{j,n}) ~ B exp(q.kbar_j + w_j),
w_j = 1/2 (pooled q^2) . sigma_j^2, gated to 0 above ln B), used on top of
"PISA: Piecewise Sparse Attention Is Wiser for Efficient Diffusion
Transformers" Section 3.2 Eq. 3-6.

The expansion is exact to second order when the key deviations of a block have
a diagonal covariance and the queries of a query block are equal; then the
mass error falls from O(eps^2) (zeroth order) to O(eps^4), which pins the 1/2,
the squared scale, the 1/n_j variance and the place where w enters."""

import math

import numpy as np
import pytest
import torch

from oracle import (block_stats, forward, gate_second_order, n_blocks, route,
                    second_order_rank_bonus, second_order_spread)


def sdpa_fp64(q, k, v, scale):
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), scale=scale)
    return o[0, 0].numpy()


def structured(eps, nb=6, B=8, d=4, seed=0):
    """Queries equal within each query block; keys = block centroid + eps times
    two orthogonal +-1 patterns in channels 0 and 1 (diagonal covariance,
    variances eps^2 a_j^2 and eps^2 b_j^2); values constant within a block."""
    rng = np.random.default_rng(seed)
    n = nb * B
    q = np.repeat(rng.standard_normal((nb, d)), B, axis=0)
    cen = rng.standard_normal((nb, d))
    amp = 0.5 + rng.random((nb, 2))
    k = np.repeat(cen, B, axis=0)
    p1 = np.tile([1.0, 1.0, -1.0, -1.0], B // 4)
    p2 = np.tile([1.0, -1.0, 1.0, -1.0], B // 4)
    for j in range(nb):
        r = slice(j * B, (j + 1) * B)
        k[r, 0] += eps * amp[j, 0] * p1
        k[r, 1] += eps * amp[j, 1] * p2
    v = np.repeat(rng.standard_normal((nb, d)), B, axis=0)
    return q, k, v, B


def slope(xs, ys):
    return np.polyfit(np.log(xs), np.log(ys), 1)[0]


def test_second_order_mass_converges_at_fourth_order():
    s = 0.8
    epss = [0.3, 0.2, 0.1, 0.05]
    e0, e2 = [], []
    for eps in epss:
        q, k, v, B = structured(eps)
        st = block_stats(q, k, v, B)
        kbar = st[1]
        w = second_order_spread(q, k, B, s)
        err0, err2 = 0.0, 0.0
        for i in range(n_blocks(len(q), B)):
            qp = s * q[i * B]
            for j in range(n_blocks(len(q), B)):
                exact = np.exp(k[j * B:(j + 1) * B] @ qp).sum()
                a = qp @ kbar[j]
                err0 = max(err0, abs(B * math.exp(a) - exact) / exact)
                err2 = max(err2, abs(B * math.exp(a + w[i, j]) - exact) / exact)
        e0.append(err0)
        e2.append(err2)
    assert 1.8 < slope(epss, e0) < 2.2, e0
    assert 3.7 < slope(epss, e2) < 4.3, e2
    assert all(b < a for a, b in zip(e0, e2))


def test_second_order_output_converges_to_dense_attention():
    """Values constant within a block make H_j = 0, so with every block
    approximated the output is the mass-weighted mean of the block values: the
    second-order output approaches dense attention at O(eps^4), the first-order
    (PISA) one at O(eps^2)."""
    s = 0.8
    epss = [0.3, 0.2, 0.1, 0.05]
    e1, e2 = [], []
    for eps in epss:
        q, k, v, B = structured(eps, seed=1)
        nb = n_blocks(len(q), B)
        ref = sdpa_fp64(q, k, v, s)
        none = [np.zeros(0, dtype=np.int64)] * nb
        o1 = forward(q, k, v, B, s, none)
        w = gate_second_order(second_order_spread(q, k, B, s), np.full(nb, B))
        o2 = forward(q, k, v, B, s, none, spread=w)
        e1.append(np.abs(o1 - ref).max())
        e2.append(np.abs(o2 - ref).max())
    assert 1.8 < slope(epss, e1) < 2.2, e1
    assert 3.6 < slope(epss, e2) < 4.4, e2


def test_spread_hand_worked_pooling():
    """d = 1, B = 2, s = 0.5, q = (1, 3, 2, 2), k = (0, 2, 5, 5): the pooled
    squared queries are (1 + 9)/2 = 5 and (4 + 4)/2 = 4 (not the squared means
    4 and 4), the key variances (0-1)^2/2 + (2-1)^2/2 = 1 and 0, so
    w = 1/2 * 0.25 * [[5*1, 5*0], [4*1, 4*0]] = [[0.625, 0], [0.5, 0]]."""
    q = np.array([[1.0], [3.0], [2.0], [2.0]])
    k = np.array([[0.0], [2.0], [5.0], [5.0]])
    w = second_order_spread(q, k, 2, 0.5)
    np.testing.assert_allclose(w, [[0.625, 0.0], [0.5, 0.0]], rtol=0, atol=1e-15)


def test_gate_uses_the_block_size_and_falls_back_to_zeroth_order():
    """w above ln(n_j) is set to 0 (not clamped); the threshold of a partial
    block of 8 tokens is ln 8, of a full block ln 64. With every spread gated
    the forward equals the plain (first-order) forward."""
    w = np.array([[2.5, 2.5, 5.0], [1.0, 4.0, 2.0]])
    g = gate_second_order(w, [64, 8, 64])
    np.testing.assert_array_equal(g, [[2.5, 0.0, 0.0], [1.0, 0.0, 2.0]])
    rng = np.random.default_rng(4)
    n, d, B = 136, 8, 64
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    nb = n_blocks(n, B)
    sets = [np.array([i], dtype=np.int64) for i in range(nb)]
    huge = np.full((nb, nb), 100.0)
    gated = gate_second_order(huge, [64, 64, 8])
    assert np.all(gated == 0.0)
    np.testing.assert_allclose(forward(q, k, v, B, 0.3, sets, spread=gated),
                               forward(q, k, v, B, 0.3, sets), rtol=0, atol=1e-15)
    small = gate_second_order(np.full((nb, nb), 0.01), [64, 64, 8])
    assert np.abs(forward(q, k, v, B, 0.3, sets, spread=small)
                  - forward(q, k, v, B, 0.3, sets)).max() > 1e-6


def test_rank_bonus_clamps_where_the_gate_zeroes():
    """The ranking bonus is min(w, ln n_j): equal to w below the limit and to
    ln n_j above it, where the forward's gated spread is 0."""
    w = np.array([[2.5, 2.5, 5.0], [1.0, 4.0, 2.0]])
    b = second_order_rank_bonus(w, [64, 8, 64])
    np.testing.assert_allclose(b, [[2.5, math.log(8), math.log(64)], [1.0, math.log(8), 2.0]],
                               rtol=0, atol=1e-15)


def test_route_with_a_pair_bonus_matches_exhaustive_search():
    """Integer scores and integer per-pair bonuses: exact fp64 ties; the
    selection must be the lexicographically first best-sum subset."""
    import itertools
    rng = np.random.default_rng(3)
    nb, topk, band = 8, 3, 1
    qbar = rng.integers(-2, 3, size=(nb, 2)).astype(np.float64)
    kbar = rng.integers(-2, 3, size=(nb, 2)).astype(np.float64)
    bonus = rng.integers(0, 3, size=(nb, nb)).astype(np.float64)
    r = qbar @ kbar.T + bonus
    sets = route(qbar, kbar, 1.0, topk, band, bonus=bonus)
    for i in range(nb):
        forced = [j for j in range(nb) if abs(i - j) <= band]
        cand = [j for j in range(nb) if j not in forced]
        best = min(itertools.combinations(cand, topk), key=lambda sub: (-sum(r[i, j] for j in sub), sub))
        assert sets[i].tolist() == sorted(forced + list(best))
