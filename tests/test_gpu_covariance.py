"""GPU parity of covariance-aware routing ("PISA: Piecewise Sparse Attention Is
Wiser for Efficient Diffusion Transformers", Section 3.3 Eq. 11 and Theorem 3.1;
Appendix D): pisa_block_heterogeneity against the oracle's M_j in both norms,
and pisa_route_covariance against the oracle's biased route.

Bars:
* M_j from the oracle's own kbar and Hbar (rounded to float32 once): within
  2e-5 of the head's largest M_j or ||H_j||_F, whichever is larger (float32
  arithmetic on a d x d product of 64 terms, then a norm; H_j - Hbar is formed
  from terms as large as H_j); from the GPU's own stats, 1e-4 of it;
* routes: identical to the oracle's except on rows whose k-th / (k+1)-th gap
  of s qbar.kbar + log(M + eps) is below 1e-5 (a near tie), which must still
  be a valid top-k within 1e-5.
"""

import numpy as np
import pytest
import torch

import oracle
from route_check import check_route_rows
from piecewise_sparse_attention_gb300.workloads import WORKLOADS, make_head, small_case

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module")
def P():
    import __graft_entry__

    __graft_entry__.build()
    from piecewise_sparse_attention_gb300 import pisa

    pisa.load()
    return pisa


def dev(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t.float()


def gpu_sets(idx, cnt):
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    return [[list(map(int, idx[h, i, : cnt[h, i]])) for i in range(idx.shape[1])]
            for h in range(idx.shape[0])]


def check_biased_route(got, qbar, kbar, scale, topk, band, bias):
    return check_route_rows(got, qbar, kbar, scale, topk, band, bias=bias)[1]


def oracle_m(q, k, v, norm):
    st = oracle.block_stats(q, k, v, 64)
    H = st[3]
    return st, oracle.block_heterogeneity(H, oracle.global_first_order(H), norm)


@pytest.mark.parametrize("norm", ["spectral", "frobenius"])
@pytest.mark.parametrize("dtype,d,n", [("bf16", 128, 1000), ("bf16", 128, 4096), ("f32", 64, 777),
                                       ("bf16", 64, 200), ("f32", 128, 50), ("bf16", 128, 64)])
def test_block_heterogeneity_parity(P, dtype, d, n, norm):
    heads = 2
    q, k, v = small_case(heads, n, d, seed=5 * n + d, dtype=dtype, spread=0.8, mean_scale=2.0)
    tk, tv = dev(k, dtype), dev(v, dtype)
    st = P.new_status()
    # (a) the kernel on the oracle's statistics, rounded to float32 once
    refs = [oracle_m(q[h], k[h], v[h], norm) for h in range(heads)]
    kb_o = torch.from_numpy(np.stack([r[0][1] for r in refs]).astype(np.float32)).cuda()
    hb_o = torch.from_numpy(np.stack([oracle.global_first_order(r[0][3])
                                      for r in refs]).astype(np.float32)).cuda()
    m_a = P.block_heterogeneity(tk, tv, kb_o, hb_o, norm=norm, status=st)
    # (b) the whole GPU chain
    _, kb, vs, _ = P.block_stats(dev(q, dtype), tk, tv, status=st)
    hbar = P.global_first_order(tk, tv, kb, vs, status=st)
    m_b = P.block_heterogeneity(tk, tv, kb, hbar, norm=norm, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    for h in range(heads):
        ref = refs[h][1]
        # float32 forms H_j - Hbar from sums as large as H_j itself, so the
        # error scales with max ||H_j|| (M_j itself may be 0: one block, H_j = Hbar)
        top = max(ref.max(), np.sqrt((refs[h][0][3] ** 2).sum(axis=(1, 2))).max())
        ga = m_a[h].cpu().double().numpy()
        gb = m_b[h].cpu().double().numpy()
        assert np.abs(ga - ref).max() <= 2e-5 * top, (np.abs(ga - ref).max(), top)
        assert np.abs(gb - ref).max() <= 1e-4 * top, (np.abs(gb - ref).max(), top)


@pytest.mark.parametrize("heads,n", [(3, 64 * 150 + 17), (5, 64 * 97), (2, 64 * 700 + 5)])
def test_frobenius_stream_many_blocks_per_cta(P, heads, n):
    """bf16, d = 128, Frobenius: the streamed kernel gives each CTA several
    consecutive (head, block) items, so these cases cross heads inside one
    CTA's range (Hbar reloaded), end heads on a ragged block and run the
    three-stage copy ring and the two accumulators through several turns.
    Every head against the oracle; repeated calls give the same bits."""
    q, k, v = small_case(heads, n, 128, seed=n + heads, dtype="bf16", spread=0.8,
                         mean_scale=2.0)
    tk, tv = dev(k, "bf16"), dev(v, "bf16")
    st = P.new_status()
    refs = [oracle_m(q[h], k[h], v[h], "frobenius") for h in range(heads)]
    kb_o = torch.from_numpy(np.stack([r[0][1] for r in refs]).astype(np.float32)).cuda()
    hb_o = torch.from_numpy(np.stack([oracle.global_first_order(r[0][3])
                                      for r in refs]).astype(np.float32)).cuda()
    m_a = P.block_heterogeneity(tk, tv, kb_o, hb_o, norm="frobenius", status=st)
    m_again = P.block_heterogeneity(tk, tv, kb_o, hb_o, norm="frobenius", status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    assert torch.equal(m_a, m_again)
    for h in range(heads):
        ref = refs[h][1]
        top = max(ref.max(), np.sqrt((refs[h][0][3] ** 2).sum(axis=(1, 2))).max())
        ga = m_a[h].cpu().double().numpy()
        assert np.abs(ga - ref).max() <= 2e-5 * top, (h, np.abs(ga - ref).max(), top)


@pytest.mark.parametrize("d,gap", [(128, 1e-4), (64, 1e-5), (128, 0.0)])
def test_spectral_norm_with_a_near_degenerate_top_pair(P, d, gap):
    """A top singular pair of H_j - Hbar split by a relative gap of `gap` (0:
    a double value) beside a random block: the Lanczos residual stop must
    still land on the largest value. f32 inputs; per block j, tokens 0-31
    carry +-1 on channel 0 in k and +-s_j in v, tokens 32-63 the same on
    channel 1 with s_j (1 - gap). The background lives on channels 2.. and is
    equal on the two tokens of each (+, -) pair, so its cross sums with the
    pattern vanish: H_j - Hbar = diag(32 (s_j - sbar), 32 (s_j - sbar)(1 - gap))
    (+) a random block, an exact pair with relative gap `gap`."""
    n = 64 * 6
    rng = np.random.default_rng(11 + d)
    k = np.zeros((1, n, d))
    v = np.zeros((1, n, d))
    k[0, :, 2:] = np.repeat(0.3 * rng.standard_normal((n // 2, d - 2)), 2, axis=0)
    v[0, :, 2:] = np.repeat(0.3 * rng.standard_normal((n // 2, d - 2)), 2, axis=0)
    sign = np.tile([1.0, -1.0], 16)
    for j in range(n // 64):
        s_j = 1.0 + 0.5 * j
        k[0, 64 * j:64 * j + 32, 0] = sign
        v[0, 64 * j:64 * j + 32, 0] = s_j * sign
        k[0, 64 * j + 32:64 * j + 64, 1] = sign
        v[0, 64 * j + 32:64 * j + 64, 1] = s_j * (1.0 - gap) * sign
    k, v = k.astype(np.float32), v.astype(np.float32)
    stx, ref = oracle_m(k[0], k[0], v[0], "spectral")
    tk, tv = dev(k, "f32"), dev(v, "f32")
    kb = torch.from_numpy(stx[1][None].astype(np.float32)).cuda()
    hb = torch.from_numpy(oracle.global_first_order(stx[3])[None].astype(np.float32)).cuda()
    st = P.new_status()
    got = P.block_heterogeneity(tk, tv, kb, hb, norm="spectral", status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    got = got[0].cpu().double().numpy()
    assert np.all(np.abs(got - ref) <= 2e-6 * ref), np.abs(got / ref - 1).max()


@pytest.mark.parametrize("gap_bits", [7, None])
def test_spectral_tc_near_degenerate_top_pair(P, gap_bits):
    """The bf16, d = 128 path (A and C = A'^T A' on the tensor cores, the
    Lanczos iteration on C) on the construction of the test above with
    bf16-exact inputs: s_j a power of two, the second direction scaled by
    1 - 2^-gap_bits (seven significant bits) or by 1 (an exact double value),
    and the background rounded to bf16 before it is used, so the oracle sees
    the very values the kernel reads. Bar 4e-6 relative: C is accumulated in
    float32 by the tensor cores, and the residual stop adds at most 5e-7."""
    d, n = 128, 64 * 6
    rng = np.random.default_rng(29)
    to_bf16 = lambda a: torch.from_numpy(a).to(torch.bfloat16).double().numpy()
    k = np.zeros((1, n, d))
    v = np.zeros((1, n, d))
    k[0, :, 2:] = np.repeat(to_bf16(0.3 * rng.standard_normal((n // 2, d - 2))), 2, axis=0)
    v[0, :, 2:] = np.repeat(to_bf16(0.3 * rng.standard_normal((n // 2, d - 2))), 2, axis=0)
    sign = np.tile([1.0, -1.0], 16)
    g = 1.0 - 2.0 ** -gap_bits if gap_bits else 1.0
    for j in range(n // 64):
        s_j = 2.0 ** (j - 2)
        k[0, 64 * j:64 * j + 32, 0] = sign
        v[0, 64 * j:64 * j + 32, 0] = s_j * sign
        k[0, 64 * j + 32:64 * j + 64, 1] = sign
        v[0, 64 * j + 32:64 * j + 64, 1] = s_j * g * sign
    assert np.array_equal(to_bf16(k), k) and np.array_equal(to_bf16(v), v)
    stx, ref = oracle_m(k[0], k[0], v[0], "spectral")
    tk, tv = dev(k, "bf16"), dev(v, "bf16")
    kb = torch.from_numpy(stx[1][None].astype(np.float32)).cuda()
    hb = torch.from_numpy(oracle.global_first_order(stx[3])[None].astype(np.float32)).cuda()
    st = P.new_status()
    got = P.block_heterogeneity(tk, tv, kb, hb, norm="spectral", status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    got = got[0].cpu().double().numpy()
    assert np.all(np.abs(got - ref) <= 4e-6 * ref), np.abs(got / ref - 1).max()


def test_spectral_and_frobenius_closed_form(P):
    """The diagonal construction of the oracle pins (d = 64, blocks of 64
    tokens): H_0 = 4 e_0 e_0^T, H_1 = 12 e_1 e_1^T, H_2 = 0."""
    d, n = 64, 192
    k = np.zeros((1, n, d), np.float32)
    v = np.zeros((1, n, d), np.float32)
    k[0, 0:64, 0] = np.tile([1, -1, 1, -1], 16) / 16.0   # sum_n a_n b_n = 4
    v[0, 0:64, 0] = np.tile([1, -1, 1, -1], 16)
    k[0, 64:128, 1] = np.tile([2, -2, 0, 0], 16) / 4.0
    v[0, 64:128, 1] = np.tile([3, -3, 0, 0], 16) / 4.0  # sum_n a_n b_n = 12
    k[0, :, 2] = 7.0
    tk, tv = dev(k, "f32"), dev(v, "f32")
    st = P.new_status()
    _, kb, vs, _ = P.block_stats(tk, tk, tv, status=st)
    hbar = P.global_first_order(tk, tv, kb, vs, status=st)
    ms = P.block_heterogeneity(tk, tv, kb, hbar, norm="spectral", status=st)
    mf = P.block_heterogeneity(tk, tv, kb, hbar, norm="frobenius", status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    np.testing.assert_allclose(ms[0].cpu().numpy(), [4, 8, 4], rtol=1e-6)
    np.testing.assert_allclose(mf[0].cpu().numpy(),
                               np.sqrt([208 / 9, 592 / 9, 160 / 9]), rtol=1e-6)


@pytest.mark.parametrize("nb,d,topk,band", [(40, 128, 5, 1), (300, 128, 17, 1), (64, 64, 100, 1),
                                             (7, 64, 3, 0), (1000, 128, 60, 2)])
def test_route_covariance_parity(P, nb, d, topk, band):
    rng = np.random.default_rng(nb + topk)
    heads = 2
    qbar = rng.standard_normal((heads, nb, d)).astype(np.float32)
    kbar = rng.standard_normal((heads, nb, d)).astype(np.float32)
    M = np.exp(1.5 * rng.standard_normal((heads, nb))).astype(np.float32)
    M[:, ::13] = 0.0  # log(eps) for some blocks
    s = 0.09
    idx, cnt = P.route_covariance(torch.from_numpy(qbar).cuda(), torch.from_numpy(kbar).cuda(),
                                  torch.from_numpy(M).cuda(), s, topk, band, eps=EPS)
    got = gpu_sets(idx, cnt)
    for h in range(heads):
        bias = oracle.covariance_bias(M[h].astype(np.float64), EPS)
        check_biased_route(got[h], qbar[h], kbar[h], s, topk, band, bias)


def test_route_covariance_integer_ties(P):
    """Integer means with a bias that is an exact float (M + eps = e^c): exact
    scores with many ties; the lowest index must win as in the oracle."""
    rng = np.random.default_rng(8)
    for nb, topk, band in [(40, 5, 1), (300, 17, 1), (64, 10, 0)]:
        qbar = rng.integers(-2, 3, size=(1, nb, 128)).astype(np.float32)
        kbar = rng.integers(-2, 3, size=(1, nb, 128)).astype(np.float32)
        M = np.ones((1, nb), np.float32)  # every bias equal: the plain route
        idx, cnt = P.route_covariance(torch.from_numpy(qbar).cuda(), torch.from_numpy(kbar).cuda(),
                                      torch.from_numpy(M).cuda(), 0.125, topk, band, eps=0.5)
        got = gpu_sets(idx, cnt)
        ora = oracle.route(qbar[0], kbar[0], 0.125, topk, band)
        assert got[0] == [list(map(int, x)) for x in ora]


def test_route_covariance_reports_bad_norms(P):
    nb = 50
    rng = np.random.default_rng(1)
    qbar = torch.from_numpy(rng.standard_normal((1, nb, 64)).astype(np.float32)).cuda()
    kbar = torch.from_numpy(rng.standard_normal((1, nb, 64)).astype(np.float32)).cuda()
    M = torch.ones(1, nb, device="cuda")
    M[0, 3] = float("nan")
    M[0, 9] = -1.0
    st = P.new_status()
    idx, cnt = P.route_covariance(qbar, kbar, M, 0.1, 4, 1, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == P.ERR_DEVICE_CHECK
    c = cnt.cpu().numpy()
    assert np.all((c >= 1) & (c <= 7))


@pytest.mark.parametrize("name,norm", [("tiny", "spectral"), ("flux", "frobenius"),
                                       ("wan", "spectral")])
def test_covariance_route_on_workloads(P, name, norm):
    """The whole covariance-aware prepare phase at the workload's launch size:
    stats, Hbar, M (both computed on the GPU), biased route; against the
    oracle's fp64 chain on the first and last heads."""
    wl = WORKLOADS[name]
    heads = [0, wl.heads - 1]
    qs, ks, vs_ = zip(*(make_head(wl, h) for h in heads))
    q, k, v = np.stack(qs), np.stack(ks), np.stack(vs_)
    tq, tk, tv = dev(q, wl.dtype), dev(k, wl.dtype), dev(v, wl.dtype)
    st = P.new_status()
    qb, kb, vs, _ = P.block_stats(tq, tk, tv, status=st)
    hbar = P.global_first_order(tk, tv, kb, vs, status=st)
    M = P.block_heterogeneity(tk, tv, kb, hbar, norm=norm, status=st)
    idx, cnt = P.route_covariance(qb, kb, M, wl.scale, wl.topk, wl.band, eps=EPS, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    got = gpu_sets(idx, cnt)
    for x in range(len(heads)):
        stx, Mref = oracle_m(q[x], k[x], v[x], norm)
        gm = M[x].cpu().double().numpy()
        top = max(Mref.max(), np.sqrt((stx[3] ** 2).sum(axis=(1, 2))).max())
        assert np.abs(gm - Mref).max() <= 1e-4 * top
        check_biased_route(got[x], stx[0], stx[1], wl.scale, wl.topk, wl.band,
                           oracle.covariance_bias(Mref, EPS))


@pytest.mark.parametrize("cov", [False, True])
def test_route_at_the_largest_block_count(P, cov):
    """n_b = 16384 (2^20 tokens), the largest the library accepts: the plain
    route and pisa_route_ex with sinks and the covariance bias (whose per-block
    bias fills the remaining shared memory), on sampled query blocks."""
    nb, d, topk, band = 16384, 64, 24, 1
    rng = np.random.default_rng(5 + cov)
    qbar = rng.standard_normal((1, nb, d)).astype(np.float32)
    kbar = rng.standard_normal((1, nb, d)).astype(np.float32)
    M = np.exp(rng.standard_normal((1, nb))).astype(np.float32) if cov else None
    n_sink = 3 if cov else 0
    st = P.new_status()
    tq, tkb = torch.from_numpy(qbar).cuda(), torch.from_numpy(kbar).cuda()
    if cov:
        idx, cnt = P.route_ex(tq, tkb, 0.125, topk, band, n_sink, mnorm=torch.from_numpy(M).cuda(),
                              eps=EPS, status=st)
    else:
        idx, cnt = P.route(tq, tkb, 0.125, topk, band, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    rows = sorted({0, 1, nb // 2, nb - 1, *rng.integers(0, nb, 12).tolist()})
    bias = oracle.covariance_bias(M[0].astype(np.float64), EPS) if cov else None
    got = [list(map(int, idx[0, i, :cnt[0, i]])) for i in rows]
    check_route_rows(got, qbar[0], kbar[0], 0.125, topk, band, bias=bias, n_sink=n_sink, rows=rows)
