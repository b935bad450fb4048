"""Pins for the hybrid-order oracle ("PISA: Piecewise Sparse Attention Is
Wiser for Efficient Diffusion Transformers", Section 3.3 Eq. 7-10, Theorem
3.1 / Appendix C Theorem C.2): it must equal the block-wise first-order result
when every block shares one H_j, differ from it by exactly q' R_t / D_t in
general, obey the Theorem C.2 bound, and reduce to dense attention at
density 1."""

import math

import numpy as np
import torch

from oracle import block_stats, forward, forward_hybrid, global_first_order, n_blocks, route


def sdpa_fp64(q, k, v, scale):
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), scale=scale)[0, 0].numpy()


def test_hybrid_equals_blockwise_when_every_block_shares_H():
    """k_{j,n} = c_j + delta_n and v_{j,n} = w_j + u_n with the same zero-mean
    delta and the same u in every block give H_j = sum_n delta_n^T u_n for all
    j, so Hbar = H_j and replacing sum alpha_j H_j by (sum alpha_j) Hbar is
    exact (Eq. 10 vs Eq. 6)."""
    B, nb, d = 16, 6, 5
    rng = np.random.default_rng(1)
    delta = rng.standard_normal((B, d))
    delta -= delta.mean(axis=0)
    u = rng.standard_normal((B, d))
    c = rng.standard_normal((nb, d)) * 2
    w = rng.standard_normal((nb, d))
    k = (c[:, None, :] + delta[None]).reshape(nb * B, d)
    v = (w[:, None, :] + u[None]).reshape(nb * B, d)
    q = rng.standard_normal((nb * B, d))
    st = block_stats(q, k, v, B)
    assert np.abs(st[3] - st[3][0]).max() < 1e-12
    for topk, band in [(0, 0), (1, 1), (2, 0)]:
        sets = route(st[0], st[1], 0.6, topk, band)
        ob = forward(q, k, v, B, 0.6, sets, stats=st)
        oh = forward_hybrid(q, k, v, B, 0.6, sets, stats=st)
        np.testing.assert_allclose(oh, ob, rtol=0, atol=1e-12)


def _alpha_and_den(q, k, v, B, s, sets, st, i):
    """Un-shifted alpha_tj over U_i and the shared denominator D_t of query
    block i, straight from the definitions (Appendix C "Notation")."""
    n, d = q.shape
    nb = n_blocks(n, B)
    rows = slice(i * B, min(i * B + B, n))
    qp = s * q[rows]
    S = set(int(j) for j in sets[i])
    U = [j for j in range(nb) if j not in S]
    alpha = np.exp(qp @ st[1][U].T)
    den = alpha @ st[4][U].astype(float)
    for j in S:
        r = slice(j * B, min(j * B + B, n))
        den = den + np.exp(qp @ k[r].T).sum(axis=1)
    return qp, U, alpha, den


def test_hybrid_error_identity_and_theorem_c2_bound():
    """Appendix C, proof of Theorem C.2: o~_t - o_t = -q' R_t / D_t with
    R_t = sum_{j in U} alpha_tj (H_j - Hbar); hence ||o~ - o|| <=
    ||q'|| M sum_U alpha / D_t (Eq. 12) with M = max_U ||H_j - Hbar||_2, and,
    with full blocks, sum_U alpha <= tau_t / B (Eq. 13)."""
    n, B, d = 160, 32, 6
    rng = np.random.default_rng(2)
    q = rng.standard_normal((n, d))
    k = rng.standard_normal((n, d)) + np.repeat(rng.standard_normal((n // B, d)), B, axis=0)
    v = rng.standard_normal((n, d))
    s = 0.5
    st = block_stats(q, k, v, B)
    Hbar = global_first_order(st[3])
    sets = route(st[0], st[1], s, 1, 0)
    ob = forward(q, k, v, B, s, sets, stats=st)
    oh = forward_hybrid(q, k, v, B, s, sets, stats=st)
    for i in range(n_blocks(n, B)):
        qp, U, alpha, den = _alpha_and_den(q, k, v, B, s, sets, st, i)
        R = np.einsum("tj,jce->tce", alpha, st[3][U] - Hbar)
        diff = oh[i * B:(i + 1) * B] - ob[i * B:(i + 1) * B]
        expect = -np.einsum("tc,tce->te", qp, R) / den[:, None]
        np.testing.assert_allclose(diff, expect, rtol=1e-9, atol=1e-12)
        M = max(np.linalg.norm(st[3][j] - Hbar, 2) for j in U)
        bound = np.linalg.norm(qp, axis=1) * M * alpha.sum(axis=1) / den
        assert np.all(np.linalg.norm(diff, axis=1) <= bound * (1 + 1e-9))
        tau = np.zeros(qp.shape[0])
        for j in U:
            r = slice(j * B, (j + 1) * B)
            tau += np.exp(qp @ k[r].T).sum(axis=1)
        assert np.all(alpha.sum(axis=1) <= tau / B * (1 + 1e-12))


def test_hybrid_density_one_is_dense_attention():
    n, B, d = 200, 32, 8
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    s = 1 / math.sqrt(d)
    st = block_stats(q, k, v, B)
    sets = route(st[0], st[1], s, 100, 1)
    np.testing.assert_allclose(forward_hybrid(q, k, v, B, s, sets, stats=st),
                               sdpa_fp64(q, k, v, s), rtol=0, atol=1e-12)


def test_hybrid_constant_values():
    """v = c: every H_j = 0 and Vhat_j = n_j c, so o = c exactly."""
    n, B, d = 100, 16, 4
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal((n, d)) * 2, rng.standard_normal((n, d)) * 2
    c = np.array([0.5, -1.0, 2.0, 0.0])
    v = np.tile(c, (n, 1))
    st = block_stats(q, k, v, B)
    sets = route(st[0], st[1], 0.7, 1, 0)
    np.testing.assert_allclose(forward_hybrid(q, k, v, B, 0.7, sets, stats=st), np.tile(c, (n, 1)),
                               rtol=0, atol=1e-13)
