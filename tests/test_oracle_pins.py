"""Pins for the fp64 oracle: each test checks it against something other than
itself (a textbook routine, a closed form, an invariant, an exact special case
or brute force), chosen so that a plausible slip (a dropped term, a wrong sign
or index, a transposed H, a missing scale, a sum in place of a mean) fails at
least one of them.

The method is the piecewise forward of "PISA: Piecewise Sparse Attention Is
Wiser for Efficient Diffusion Transformers", Section 3.2, Eq. (3)-(6), with the
error analysis of Appendix C.
"""

import itertools
import math

import numpy as np
import pytest
import torch

from oracle import block_stats, forward, forward_head, n_blocks, route, route_gaps


def sdpa_fp64(q, k, v, scale):
    """Dense softmax attention, Eq. (1), via PyTorch's CPU routine in fp64."""
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), scale=scale)
    return o[0, 0].numpy()


def rand(n, d, seed, mean=0.0):
    rng = np.random.default_rng(seed)
    return (mean + rng.standard_normal((n, d)),
            mean + rng.standard_normal((n, d)),
            rng.standard_normal((n, d)))


@pytest.mark.parametrize("n,B,d", [(256, 64, 16), (200, 32, 8), (37, 16, 4), (5, 16, 3)])
def test_density_one_is_dense_attention(n, B, d):
    """Every block selected (U_i empty) leaves only the exact term: the output is
    dense softmax attention (Eq. (1)); cf. the README's density=1.0 check."""
    q, k, v = rand(n, d, 1)
    s = 0.7 / math.sqrt(d)
    nb = n_blocks(n, B)
    o, sets, _ = forward_head(q, k, v, B, s, topk=nb, band=1)
    assert all(len(S) == nb for S in sets)
    np.testing.assert_allclose(o, sdpa_fp64(q, k, v, s), rtol=0, atol=1e-12)


@pytest.mark.parametrize("n,B", [(256, 64), (100, 16)])
def test_identical_keys_make_taylor_exact(n, B):
    """Keys equal within each block: H_j = 0 and n_j exp(q'.kbar_j) equals the
    exact block sum, so any routing gives dense attention (zeroth-order term of
    Eq. (3)/(5) pinned, including the n_j of a partial last block)."""
    d = 8
    rng = np.random.default_rng(2)
    nb = n_blocks(n, B)
    centers = rng.standard_normal((nb, d)) * 2
    k = np.repeat(centers, B, axis=0)[:n]
    q = rng.standard_normal((n, d)) * 2
    v = rng.standard_normal((n, d))
    s = 1 / math.sqrt(d)
    for topk, band in [(0, 0), (1, 0), (2, 1)]:
        o, _, st = forward_head(q, k, v, B, s, topk, band)
        assert np.abs(st[3]).max() < 1e-12
        np.testing.assert_allclose(o, sdpa_fp64(q, k, v, s), rtol=0, atol=1e-12)


def test_deviation_orthogonal_to_queries_is_exact():
    """Key deviations orthogonal to every query: exp(q'.k_{j,n}) = exp(q'.kbar_j)
    for all n and the first-order term q' H_j vanishes, so the approximation is
    exact while H_j itself is non-zero."""
    n, B, d = 192, 64, 8
    rng = np.random.default_rng(3)
    nb = n_blocks(n, B)
    q = np.zeros((n, d))
    q[:, :4] = rng.standard_normal((n, 4))
    centers = np.zeros((nb, d))
    centers[:, :4] = rng.standard_normal((nb, 4))
    dev = np.zeros((n, d))
    dev[:, 4:] = rng.standard_normal((n, 4))
    k = np.repeat(centers, B, axis=0)[:n] + dev
    v = rng.standard_normal((n, d))
    s = 0.5
    o, _, st = forward_head(q, k, v, B, s, topk=0, band=0)
    assert np.abs(st[3]).max() > 1e-2
    np.testing.assert_allclose(o, sdpa_fp64(q, k, v, s), rtol=0, atol=1e-12)


def test_first_order_term_gives_second_order_error():
    """Keys k = kbar_j + eps * delta: the block-wise first-order expansion
    leaves an O(eps^2) error against dense attention while the zeroth-order
    variant leaves O(eps) (Appendix C, remark 3: Lagrange remainder). A wrong
    sign, scale or orientation of the q' H_j term turns the slope back to 1."""
    n, B, d = 128, 32, 6
    rng = np.random.default_rng(4)
    nb = n_blocks(n, B)
    centers = rng.standard_normal((nb, d))
    delta = rng.standard_normal((n, d))
    delta -= np.repeat(delta.reshape(nb, B, d).mean(axis=1), B, axis=0)
    q = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d)) + 0.3
    s = 0.8
    errs1, errs0 = [], []
    eps_list = [1e-1, 3e-2, 1e-2, 3e-3]
    for eps in eps_list:
        k = np.repeat(centers, B, axis=0) + eps * delta
        st = block_stats(q, k, v, B)
        sets = route(st[0], st[1], s, topk=0, band=0)
        ref = sdpa_fp64(q, k, v, s)
        errs1.append(np.abs(forward(q, k, v, B, s, sets, stats=st) - ref).max())
        errs0.append(np.abs(forward(q, k, v, B, s, sets, stats=st, first_order=False) - ref).max())
    x = np.log(eps_list)
    slope1 = np.polyfit(x, np.log(errs1), 1)[0]
    slope0 = np.polyfit(x, np.log(errs0), 1)[0]
    assert 1.85 < slope1 < 2.15, (slope1, errs1)
    assert 0.9 < slope0 < 1.1, (slope0, errs0)


def test_first_order_term_is_the_derivative():
    """The U-block numerator of Eq. (5)+(6) is exp(a)(Vhat + q'H): its part
    linear in the key deviations must equal the derivative at eps = 0 of the
    exact block numerator sum_n exp(q'.(kbar + eps delta_n)) v_n, taken by a
    central difference (an independent route to the same quantity)."""
    B, d = 16, 5
    rng = np.random.default_rng(5)
    kbar = rng.standard_normal(d)
    delta = rng.standard_normal((B, d))
    delta -= delta.mean(axis=0)
    v = rng.standard_normal((B, d))
    qp = 0.6 * rng.standard_normal(d)
    h = 1e-5

    def exact_num(eps):
        kk = kbar + eps * delta
        return (np.exp(kk @ qp)[:, None] * v).sum(axis=0)

    deriv = (exact_num(h) - exact_num(-h)) / (2 * h)
    k = kbar + delta
    _, _, vsum, H, _ = block_stats(np.zeros((B, d)), k, v, B)
    first = math.exp(qp @ kbar) * (qp @ H[0])
    np.testing.assert_allclose(first, deriv, rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(math.exp(qp @ kbar) * vsum[0], exact_num(0.0), rtol=1e-13)


def test_linearisation_identity():
    """q' H_j = sum_n (q'.k_{j,n} - q'.kbar_j) v_{j,n}: fixes the orientation
    (key channel x value channel) and the centring of H_j."""
    n, B, d = 150, 64, 7
    q, k, v = rand(n, d, 6, mean=0.5)
    qbar, kbar, vsum, H, nj = block_stats(q, k, v, B)
    qp = 0.3 * q[:10]
    for j in range(n_blocks(n, B)):
        r = slice(j * B, min(j * B + B, n))
        direct = ((qp @ k[r].T) - (qp @ kbar[j])[:, None]) @ v[r]
        np.testing.assert_allclose(qp @ H[j], direct, rtol=1e-12, atol=1e-12)


def test_global_first_order_identity():
    """sum_j H_j = K^T V - sum_j n_j kbar_j (x) vbar_j (the identity the
    Piecewise-Taylor-Attention README uses for its hc-free statistics); also
    pins mean-vs-sum for kbar and Vhat."""
    n, B, d = 300, 64, 6
    q, k, v = rand(n, d, 7, mean=1.0)
    qbar, kbar, vsum, H, nj = block_stats(q, k, v, B)
    vbar = vsum / nj[:, None]
    rhs = k.T @ v - sum(nj[j] * np.outer(kbar[j], vbar[j]) for j in range(len(nj)))
    np.testing.assert_allclose(H.sum(axis=0), rhs, rtol=1e-12, atol=1e-11)
    np.testing.assert_allclose(nj.sum(), n)
    np.testing.assert_allclose((kbar * nj[:, None]).sum(axis=0), k.sum(axis=0), rtol=1e-12)
    np.testing.assert_allclose(vsum.sum(axis=0), v.sum(axis=0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose((qbar * nj[:, None]).sum(axis=0), q.sum(axis=0), rtol=1e-12)


def test_constant_values_give_constant_output():
    """v = c everywhere: H_j = 0, Vhat_j = n_j c, so numerator = c x denominator
    and o = c for any routing (exact and approximate masses must match)."""
    n, B, d = 130, 32, 5
    q, k, _ = rand(n, d, 8)
    c = np.array([1.5, -2.0, 0.25, 3.0, 0.0])
    v = np.tile(c, (n, 1))
    for topk, band in [(0, 0), (1, 1), (3, 0)]:
        o, _, _ = forward_head(q * 3, k * 3, v, B, 0.4, topk, band)
        np.testing.assert_allclose(o, np.tile(c, (n, 1)), rtol=0, atol=1e-13)


def test_jensen_block_mass_lower_bound():
    """Appendix C, Eq. (13): exp(q'.kbar_j) <= (1/n_j) sum_n exp(q'.k_{j,n})
    for every query and block, i.e. the zeroth-order mass never exceeds the
    true block mass."""
    from piecewise_sparse_attention_gb300.workloads import WORKLOADS, make_inputs

    wl = WORKLOADS["tiny"]
    q, k, v = make_inputs(wl, heads=[0])
    q, k = q[0].astype(np.float64), k[0].astype(np.float64)
    _, kbar, _, _, nj = block_stats(q, k, v[0], wl.block)
    qp = wl.scale * q[::7]
    for j in range(len(nj)):
        r = slice(j * wl.block, min((j + 1) * wl.block, len(k)))
        exact = np.exp(qp @ k[r].T).sum(axis=1)
        approx = nj[j] * np.exp(qp @ kbar[j])
        assert np.all(approx <= exact * (1 + 1e-14))


def test_within_block_permutation_invariance():
    """Reordering the key/value rows inside each key block leaves every output
    unchanged (block statistics and exact block sums are order-free)."""
    n, B, d = 200, 32, 6
    q, k, v = rand(n, d, 9)
    rng = np.random.default_rng(10)
    perm = np.arange(n)
    for j in range(n_blocks(n, B)):
        r = np.arange(j * B, min(j * B + B, n))
        perm[r] = rng.permutation(r)
    o1, s1, _ = forward_head(q, k, v, B, 0.5, 2, 1)
    o2, s2, _ = forward_head(q, k[perm], v[perm], B, 0.5, 2, 1)
    assert all(np.array_equal(a, b) for a, b in zip(s1, s2))
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def _brute_force_sets(r, topk, band):
    """Enumerate every k-subset of the non-band blocks; keep those of maximal
    score sum and take the lexicographically smallest sorted tuple (lowest
    index wins ties)."""
    nb = r.shape[0]
    out = []
    for i in range(nb):
        in_band = [j for j in range(nb) if abs(i - j) <= band]
        cand = [j for j in range(nb) if abs(i - j) > band]
        kk = min(topk, len(cand))
        best, best_key = None, None
        for sub in itertools.combinations(cand, kk):
            total = sum(r[i, j] for j in sub)
            key = (-total, sub)
            if best_key is None or key < best_key:
                best, best_key = sub, key
        out.append(sorted(in_band + list(best)))
    return out


@pytest.mark.parametrize("nb,d,topk,band,seed", [
    (7, 3, 2, 1, 0), (8, 2, 3, 0, 1), (6, 2, 1, 1, 2), (9, 3, 2, 2, 3),
    (5, 2, 0, 1, 4), (6, 2, 5, 1, 5), (4, 1, 1, 0, 6)])
def test_route_matches_brute_force_with_ties(nb, d, topk, band, seed):
    """Small integer block means give exact fp64 scores with many ties; the
    sort-based selection must equal exhaustive search with the lowest-index
    tie-break (Algorithm 1 step 2; the README's band knob)."""
    rng = np.random.default_rng(seed)
    qbar = rng.integers(-2, 3, size=(nb, d)).astype(np.float64)
    kbar = rng.integers(-2, 3, size=(nb, d)).astype(np.float64)
    sets = route(qbar, kbar, 1.0, topk, band)
    r = qbar @ kbar.T
    expect = _brute_force_sets(r, topk, band)
    for i in range(nb):
        assert list(sets[i]) == expect[i], (i, sets[i], expect[i])


def test_route_edges():
    """Band clipped at the first/last block; top-k = 0 keeps only the band;
    top-k beyond the candidate count selects everything."""
    nb, d = 10, 4
    rng = np.random.default_rng(11)
    qbar, kbar = rng.standard_normal((nb, d)), rng.standard_normal((nb, d))
    s0 = route(qbar, kbar, 0.5, 0, 1)
    assert list(s0[0]) == [0, 1] and list(s0[nb - 1]) == [nb - 2, nb - 1]
    assert list(s0[4]) == [3, 4, 5]
    sall = route(qbar, kbar, 0.5, 100, 1)
    assert all(list(S) == list(range(nb)) for S in sall)
    s2 = route(qbar, kbar, 0.5, 2, 0)
    r = qbar @ kbar.T
    for i in range(nb):
        cand = [j for j in range(nb) if j != i]
        best = sorted(cand, key=lambda j: -r[i, j])[:2]
        assert list(s2[i]) == sorted([i] + best)
    g = route_gaps(qbar, kbar, 0.5, 2, 0)
    assert np.all(g > 0) and np.all(np.isfinite(g))
    assert np.all(np.isinf(route_gaps(qbar, kbar, 0.5, 100, 0)))


def test_all_approximate_matches_hand_evaluation():
    """Every block approximated (empty S_i): o_t = sum_j alpha_j (Vhat_j + q'H_j)
    / sum_j n_j alpha_j, evaluated here token by token in its expanded form
    alpha_j (1 + q'.(k_{j,n} - kbar_j)) v_{j,n} with math.exp on a ragged case."""
    n, B, d = 11, 4, 2
    q, k, v = rand(n, d, 12)
    s = 0.9
    nb = n_blocks(n, B)
    o = forward(q, k, v, B, s, [np.zeros(0, np.int64)] * nb)
    for t in range(n):
        num = np.zeros(d)
        den = 0.0
        for j in range(nb):
            rows = range(j * B, min(j * B + B, n))
            kb = [sum(k[r][c] for r in rows) / len(rows) for c in range(d)]
            a = math.exp(s * sum(q[t][c] * kb[c] for c in range(d)))
            den += len(rows) * a
            for r in rows:
                lin = s * sum(q[t][c] * (k[r][c] - kb[c]) for c in range(d))
                num += a * (1.0 + lin) * v[r]
        np.testing.assert_allclose(o[t], num / den, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("seed,nb,d,topk,band,n_sink,extra", [
    (31, 9, 3, 2, 0, 0, None), (32, 12, 2, 3, 1, 0, None), (33, 10, 4, 1, 2, 2, "bias"),
    (34, 11, 3, 4, 1, 1, "bonus"), (35, 7, 2, 5, 1, 0, None), (36, 13, 3, 0, 1, 0, None),
    (37, 8, 2, 2, 0, 3, "bias")])
def test_route_gaps_brute_force(seed, nb, d, topk, band, n_sink, extra):
    """The selection margin checked against a definition that sorts nothing:
    scores summed by explicit loops, the free candidates the route did pick and
    those it did not, margin = (lowest picked score) - (highest unpicked score);
    inf when either side is empty. Scores are on a coarse grid, so ties at the
    boundary (margin 0) occur."""
    rng = np.random.default_rng(seed)
    qbar = rng.integers(-2, 3, size=(nb, d)).astype(np.float64)
    kbar = rng.integers(-2, 3, size=(nb, d)).astype(np.float64)
    s = 0.75
    bias = rng.integers(-2, 3, size=nb) * 0.5 if extra == "bias" else None
    bonus = rng.integers(0, 3, size=(nb, nb)) * 0.25 if extra == "bonus" else None
    sets = route(qbar, kbar, s, topk, band, bias=bias, n_sink=n_sink, bonus=bonus)
    gaps = route_gaps(qbar, kbar, s, topk, band, bias=bias, n_sink=n_sink, bonus=bonus)
    ties = 0
    for i in range(nb):
        score = []
        for j in range(nb):
            x = s * sum(qbar[i][c] * kbar[j][c] for c in range(d))
            x += 0.0 if bias is None else bias[j]
            x += 0.0 if bonus is None else bonus[i][j]
            score.append(x)
        free = [j for j in range(nb) if abs(i - j) > band and j >= n_sink]
        picked = [j for j in free if j in set(sets[i].tolist())]
        rest = [j for j in free if j not in picked]
        assert len(picked) == min(topk, len(free))
        if picked and rest:
            want = min(score[j] for j in picked) - max(score[j] for j in rest)
            assert gaps[i] == pytest.approx(want, abs=1e-12), (i, gaps[i], want)
            ties += want == 0
        else:
            assert gaps[i] == np.inf, (i, gaps[i])
    if seed in (31, 32, 33):
        assert ties > 0, "this seed's grid has boundary ties"
