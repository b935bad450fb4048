"""Pins for the oracle's covariance-aware routing ("PISA: Piecewise Sparse
Attention Is Wiser for Efficient Diffusion Transformers", Section 3.3
"Covariance-Aware Block Selection", Eq. 11, Theorem 3.1; Appendix D Eq. 14):
the per-block heterogeneity M_j = ||H_j - Hbar|| against hand-derived closed
forms and an independent power iteration, and the biased route against
exhaustive search and the invariances the pages state."""

import itertools
import math

import numpy as np
import pytest

from oracle import block_heterogeneity, block_stats, covariance_bias, route, route_gaps


def _stats(k, v, B):
    q = np.zeros_like(k)
    return block_stats(q, k, v, B)


def test_rank_one_heterogeneity_closed_form():
    """Block 0's keys deviate from their mean only in channel 1, by
    a = (1, -1, 2, -2); blocks 1 and 2 have identical keys (H_1 = H_2 = 0).
    Then H_0 = e_1 (x) w with w = sum_n a_n v_n = (3, 5, -1), Hbar = H_0 / 3, and
    both norms of H_0 - Hbar are (2/3)|w|, of H_1 - Hbar and H_2 - Hbar (1/3)|w|."""
    B, d = 4, 3
    k = np.zeros((12, d))
    k[0:4] = [0.5, 0.0, -1.0]
    k[0:4, 1] += [1, -1, 2, -2]
    k[4:8] = [2.0, 1.0, 0.0]
    k[8:12] = [-1.0, 3.0, 1.0]
    v = np.zeros((12, d))
    v[0:4] = [[1, 0, 2], [0, 1, 1], [2, 2, 0], [1, -1, 1]]
    v[4:12] = np.arange(24).reshape(8, 3) % 5  # anything: their keys do not deviate
    _, _, _, H, _ = _stats(k, v, B)
    Hbar = H.mean(axis=0)
    w = np.sqrt(35.0)
    for norm in ("spectral", "frobenius"):
        M = block_heterogeneity(H, Hbar, norm)
        np.testing.assert_allclose(M, [2 * w / 3, w / 3, w / 3], rtol=1e-14)


def test_spectral_and_frobenius_differ_on_diagonal_blocks():
    """H_0 = 4 e_0 e_0^T (deviations a = (1,-1,1,-1) in key channel 0, values a
    in value channel 0), H_1 = 12 e_1 e_1^T (a = (2,-2,0,0), values (3,-3,0,0)
    in channel 1), H_2 = 0, so Hbar = diag(4/3, 4, 0) and H_j - Hbar is diagonal:
    diag(8/3, -4), diag(-4/3, 8), diag(-4/3, -4). The spectral norm is the
    largest |entry|, the Frobenius norm the root of the sum of squares."""
    B, d = 4, 3
    k = np.zeros((12, d))
    v = np.zeros((12, d))
    k[0:4, 0] = [1, -1, 1, -1]
    v[0:4, 0] = [1, -1, 1, -1]
    k[4:8, 1] = [2, -2, 0, 0]
    v[4:8, 1] = [3, -3, 0, 0]
    k[:, 2] = 7.0  # a constant channel deviates nowhere
    _, _, _, H, _ = _stats(k, v, B)
    Hbar = H.mean(axis=0)
    np.testing.assert_allclose(block_heterogeneity(H, Hbar, "spectral"), [4, 8, 4], rtol=1e-14)
    np.testing.assert_allclose(block_heterogeneity(H, Hbar, "frobenius"),
                               [math.sqrt(208 / 9), math.sqrt(592 / 9), math.sqrt(160 / 9)],
                               rtol=1e-14)


def test_spectral_norm_matches_power_iteration_and_norm_inequalities():
    """On random blocks: the spectral norm equals sqrt of the limit of a power
    iteration on A^T A (an independent algorithm), and
    max|a_ce| <= ||A||_2 <= ||A||_F <= sqrt(d) ||A||_2."""
    rng = np.random.default_rng(3)
    B, d, nb = 8, 5, 6
    k = rng.standard_normal((B * nb, d))
    v = rng.standard_normal((B * nb, d))
    _, _, _, H, _ = _stats(k, v, B)
    Hbar = H.mean(axis=0)
    ms = block_heterogeneity(H, Hbar, "spectral")
    mf = block_heterogeneity(H, Hbar, "frobenius")
    for j in range(nb):
        A = H[j] - Hbar
        x = np.ones(d)
        for _ in range(5000):
            x = A.T @ (A @ x)
            x /= np.linalg.norm(x)
        np.testing.assert_allclose(ms[j], np.linalg.norm(A @ x), rtol=1e-10)
        assert np.abs(A).max() <= ms[j] * (1 + 1e-12)
        assert ms[j] <= mf[j] * (1 + 1e-12)
        assert mf[j] <= math.sqrt(d) * ms[j] * (1 + 1e-12)


def test_identical_blocks_have_zero_heterogeneity():
    """Every block a copy of the same tokens: all H_j equal Hbar, M_j = 0, and
    the bias is log(eps) for every block (Eq. 11's eps keeps it finite)."""
    rng = np.random.default_rng(5)
    kb, vb = rng.standard_normal((8, 4)), rng.standard_normal((8, 4))
    k, v = np.tile(kb, (5, 1)), np.tile(vb, (5, 1))
    _, _, _, H, _ = _stats(k, v, 8)
    for norm in ("spectral", "frobenius"):
        M = block_heterogeneity(H, H.mean(axis=0), norm)
        assert np.abs(M).max() < 1e-12
    np.testing.assert_allclose(covariance_bias(np.zeros(3), 1e-6), np.full(3, math.log(1e-6)))


def _brute_force_sets(r, topk, band):
    nb = r.shape[0]
    out = []
    for i in range(nb):
        in_band = [j for j in range(nb) if abs(i - j) <= band]
        cand = [j for j in range(nb) if abs(i - j) > band]
        kk = min(topk, len(cand))
        best_key, best = None, None
        for sub in itertools.combinations(cand, kk):
            key = (-sum(r[i, j] for j in sub), sub)
            if best_key is None or key < best_key:
                best_key, best = key, sub
        out.append(sorted(in_band + list(best)))
    return out


@pytest.mark.parametrize("nb,d,topk,band,seed", [(7, 3, 2, 1, 0), (8, 2, 3, 0, 1),
                                                  (9, 3, 2, 2, 3), (6, 2, 4, 1, 4)])
def test_biased_route_matches_brute_force_with_ties(nb, d, topk, band, seed):
    """Integer means and integer biases give exact fp64 scores with many ties;
    the selection by s q.k + bias must equal exhaustive search over subsets
    with the lowest-index tie-break."""
    rng = np.random.default_rng(seed)
    qbar = rng.integers(-2, 3, size=(nb, d)).astype(np.float64)
    kbar = rng.integers(-2, 3, size=(nb, d)).astype(np.float64)
    bias = rng.integers(-2, 3, size=nb).astype(np.float64)
    sets = route(qbar, kbar, 1.0, topk, band, bias=bias)
    expect = _brute_force_sets(qbar @ kbar.T + bias[None, :], topk, band)
    assert [list(x) for x in sets] == expect


def test_bias_shift_and_mean_normalisation_do_not_change_the_route():
    """Eq. 11 and Eq. 14 differ by -log(Mbar), the same for every block, and
    the softmax is monotone: adding a constant to every bias leaves every S_i
    unchanged. A zero-spread bias gives the plain route."""
    rng = np.random.default_rng(11)
    nb, d = 24, 8
    qbar, kbar = rng.standard_normal((nb, d)), rng.standard_normal((nb, d))
    M = np.exp(rng.standard_normal(nb))
    b = covariance_bias(M, 1e-6)
    a = route(qbar, kbar, 0.3, 5, 1, bias=b)
    c = route(qbar, kbar, 0.3, 5, 1, bias=b - math.log(M.mean()))
    assert all(np.array_equal(x, y) for x, y in zip(a, c))
    p = route(qbar, kbar, 0.3, 5, 1)
    z = route(qbar, kbar, 0.3, 5, 1, bias=np.full(nb, 2.5))
    assert all(np.array_equal(x, y) for x, y in zip(p, z))


def test_dominant_heterogeneity_forces_selection():
    """A block whose M_j dominates every score difference is chosen by every
    query block for which it is a candidate (the covariance prior keeps the
    blocks the global first order would approximate worst); a block with a
    very small M_j is chosen by none unless there is nothing else to take."""
    rng = np.random.default_rng(2)
    nb, d = 16, 4
    qbar, kbar = rng.standard_normal((nb, d)), rng.standard_normal((nb, d))
    M = np.ones(nb)
    M[9] = 1e30
    M[3] = 1e-30
    b = covariance_bias(M, 0.0)
    sets = route(qbar, kbar, 0.5, 3, 1, bias=b)
    for i, s in enumerate(sets):
        if abs(i - 9) > 1:
            assert 9 in s
        if abs(i - 3) > 1:
            assert 3 not in s
    gaps = route_gaps(qbar, kbar, 0.5, 3, 1, bias=b)
    assert np.all(gaps > 0)
