"""GPU parity of the second-order block mass (Piecewise-Taylor-Attention
README, "Blog post"; on top of "PISA: Piecewise Sparse Attention Is Wiser for
Efficient Diffusion Transformers" Section 3.2 Eq. 3-6): pisa_second_order_spread
and pisa_forward_second_order against the oracle.

Bars: qsq and kvar within 1e-5 relative (float32 sums of <= 64 terms); w within
2e-5 * max(1, w) where the gate decision is clear; entries within 1e-4 of the
gate ln n_j may be decided either way (the decision is taken on the float32
value) and the oracle then uses the GPU's decision; outputs as for
pisa_forward (f32: max-abs 1e-4; bf16: max-abs 2e-2 and row cosine 0.9999).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from route_check import check_route_rows
from piecewise_sparse_attention_gb300.workloads import WORKLOADS, make_head, small_case

pytestmark = pytest.mark.gpu

NEAR = 1e-4


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


def check_output(got, ref, in_dtype):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref).max()
    if in_dtype == "f32":
        assert err <= 1e-4, err
    else:
        cos = (got * ref).sum(1) / (np.linalg.norm(got, axis=1) * np.linalg.norm(ref, axis=1) + 1e-300)
        assert err <= 2e-2, err
        assert cos.min() >= 0.9999, cos.min()


def oracle_spread(q, k, scale, gw):
    """The oracle's gated spread, taking the GPU's decision (gw == 0 or not)
    on entries within NEAR of the gate. Also checks the clear entries."""
    n = len(q)
    nb = -(-n // 64)
    nj = np.array([min(64, n - 64 * j) for j in range(nb)])
    w = oracle.second_order_spread(q, k, 64, scale)
    lim = np.log(nj.astype(np.float64))[None, :]
    near = np.abs(w - lim) < NEAR
    g = oracle.gate_second_order(w, nj)
    clear = ~near
    assert np.all(np.abs(gw[clear] - g[clear]) <= 2e-5 * np.maximum(1.0, np.abs(g[clear]))), \
        np.abs(gw[clear] - g[clear]).max()
    g[near] = np.where(gw[near] == 0.0, 0.0, w[near])
    return g


@pytest.mark.parametrize("dtype,d,n,spread", [("bf16", 128, 1000, 0.6), ("bf16", 128, 4096, 1.4),
                                              ("f32", 64, 777, 1.0), ("bf16", 64, 200, 2.0),
                                              ("f32", 128, 50, 0.8)])
def test_second_order_spread_parity(P, dtype, d, n, spread):
    heads = 2
    q, k, v = small_case(heads, n, d, seed=11 * n + d, dtype=dtype, spread=spread, mean_scale=1.5)
    tq, tk, tv = dev(q, dtype), dev(k, dtype), dev(v, dtype)
    st = P.new_status()
    _, kb, _, _ = P.block_stats(tq, tk, tv, status=st)
    s = 1 / math.sqrt(d)
    w, qsq, kvar = P.second_order_spread(tq, tk, kb, s, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    nb = -(-n // 64)
    gated_any = False
    for h in range(heads):
        rq = np.stack([(q[h][i * 64:(i + 1) * 64].astype(np.float64) ** 2).mean(0) for i in range(nb)])
        rk = np.stack([k[h][j * 64:(j + 1) * 64].astype(np.float64).var(0) for j in range(nb)])
        np.testing.assert_allclose(qsq[h].cpu().double().numpy(), rq, rtol=1e-5, atol=1e-12)
        np.testing.assert_allclose(kvar[h].cpu().double().numpy(), rk, rtol=1e-5, atol=1e-9)
        gw = w[h].cpu().double().numpy()
        oracle_spread(q[h], k[h], s, gw)
        gated_any |= bool((gw == 0).any())
    if spread >= 1.4:
        assert gated_any  # the gate is exercised


@pytest.mark.parametrize("dtype,d,n,topk,band,spread", [
    ("bf16", 128, 1000, 3, 1, 0.6), ("bf16", 128, 4096, 11, 1, 1.0), ("bf16", 128, 777, 2, 0, 1.4),
    ("bf16", 64, 1000, 3, 1, 0.8), ("f32", 64, 1000, 4, 1, 0.7), ("f32", 128, 333, 2, 2, 1.2),
    ("bf16", 128, 64, 0, 0, 1.0)])
def test_forward_second_order_parity(P, dtype, d, n, topk, band, spread):
    heads = 2
    q, k, v = small_case(heads, n, d, seed=n + 3 * topk, dtype=dtype, spread=spread, mean_scale=1.2)
    tq, tk, tv = dev(q, dtype), dev(k, dtype), dev(v, dtype)
    s = 1 / math.sqrt(d)
    st = P.new_status()
    qb, kb, _, _ = P.block_stats(tq, tk, tv, status=st)
    w, _, _ = P.second_order_spread(tq, tk, kb, s, status=st)
    idx, cnt = P.route(qb, kb, s, topk, band, status=st)
    out = P.forward_second_order(tq, tk, tv, idx, cnt, w, s, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    idx, cnt, out = idx.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()
    for h in range(heads):
        sets = [idx[h, i, :cnt[h, i]].astype(np.int64) for i in range(idx.shape[1])]
        ref_w = oracle_spread(q[h], k[h], s, w[h].cpu().double().numpy())
        ref = oracle.forward(q[h], k[h], v[h], 64, s, sets, spread=ref_w)
        check_output(out[h], ref, dtype)


@pytest.mark.parametrize("name", ["tiny", "flux", "wan"])
def test_forward_second_order_workloads(P, name):
    """The whole second-order chain at the workload's launch size (GPU stats,
    spread, route, forward); the oracle on the GPU's route and gate decisions,
    sampled query blocks for the large workloads."""
    wl = WORKLOADS[name]
    heads = list(range(wl.heads)) if name == "tiny" else [0, wl.heads - 1]
    qs, ks, vs = zip(*(make_head(wl, h) for h in heads))
    q, k, v = np.stack(qs), np.stack(ks), np.stack(vs)
    tq, tk, tv = dev(q, wl.dtype), dev(k, wl.dtype), dev(v, wl.dtype)
    st = P.new_status()
    qb, kb, _, _ = P.block_stats(tq, tk, tv, status=st)
    w, _, _ = P.second_order_spread(tq, tk, kb, wl.scale, status=st)
    idx, cnt = P.route(qb, kb, wl.scale, wl.topk, wl.band, status=st)
    out = P.forward_second_order(tq, tk, tv, idx, cnt, w, wl.scale, out_dtype=torch.float32,
                                 status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    idx, cnt, out = idx.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()
    rng = np.random.default_rng(9)
    for x in range(len(heads)):
        sets = [idx[x, i, :cnt[x, i]].astype(np.int64) for i in range(wl.nb)]
        ref_w = oracle_spread(q[x], k[x], wl.scale, w[x].cpu().double().numpy())
        blocks = None if wl.nb <= 72 else sorted({0, wl.nb - 1, *rng.integers(1, wl.nb - 1, 6).tolist()})
        ref = oracle.forward(q[x], k[x], v[x], wl.block, wl.scale, sets, spread=ref_w,
                             qblocks=blocks)
        if blocks is None:
            check_output(out[x], ref, wl.dtype)
        else:
            for i in blocks:
                rows = slice(i * wl.block, min((i + 1) * wl.block, wl.n))
                check_output(out[x][rows], ref[i], wl.dtype)




@pytest.mark.parametrize("name,extra", [("flux", "none"), ("wan", "none"), ("flux", "cov_sinks")])
def test_route_with_rank_bonus(P, name, extra):
    """pisa_route_ex with the second-order ranking bonus min(w, ln n_j) (the
    README's router) against the oracle's fp64 route with its own bonus; the
    bonus is continuous, so only near ties (gap < 1e-5) may differ."""
    wl = WORKLOADS[name]
    heads = [0, wl.heads - 1]
    qs, ks, vs = zip(*(make_head(wl, h) for h in heads))
    q, k, v = np.stack(qs), np.stack(ks), np.stack(vs)
    tq, tk, tv = dev(q, wl.dtype), dev(k, wl.dtype), dev(v, wl.dtype)
    st = P.new_status()
    qb, kb, vsum, _ = P.block_stats(tq, tk, tv, status=st)
    _, _, _, wrank = P.second_order_spread(tq, tk, kb, wl.scale, with_rank=True, status=st)
    n_sink = 2 if extra == "cov_sinks" else 0
    M = None
    if extra == "cov_sinks":
        hbar = P.global_first_order(tk, tv, kb, vsum, status=st)
        M = P.block_heterogeneity(tk, tv, kb, hbar, norm="frobenius", status=st)
    idx, cnt = P.route_ex(qb, kb, wl.scale, wl.topk, wl.band, n_sink, mnorm=M, bonus=wrank,
                          status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    nb = wl.nb
    nj = np.array([min(64, wl.n - 64 * j) for j in range(nb)])
    for x in range(len(heads)):
        sto = oracle.block_stats(q[x], k[x], v[x], 64)
        bonus = oracle.second_order_rank_bonus(oracle.second_order_spread(q[x], k[x], 64, wl.scale), nj)
        bias = None
        if M is not None:
            H = sto[3]
            bias = oracle.covariance_bias(oracle.block_heterogeneity(H, oracle.global_first_order(H),
                                                                     "frobenius"), 1e-6)
        got = [list(map(int, idx[x, i, :cnt[x, i]])) for i in range(nb)]
        check_route_rows(got, sto[0], sto[1], wl.scale, wl.topk, wl.band, bias=bias, n_sink=n_sink,
                         bonus=bonus)
