"""GPU parity of the Morton reorder, the fused head gather / restore and sink
blocks (Piecewise-Taylor-Attention README: "Morton tile reorder + fused gather
kernel", n_sink_blocks; routing of "PISA: Piecewise Sparse Attention Is Wiser
for Efficient Diffusion Transformers", Algorithm 1 step 2).

Bars: permutations and copies bit-exact; routes as pisa_route (identical except
at near ties below 1e-5); outputs as pisa_forward."""

import math

import numpy as np
import pytest
import torch

import oracle
from route_check import check_route_rows
from piecewise_sparse_attention_gb300.workloads import WORKLOADS, make_head

pytestmark = pytest.mark.gpu



@pytest.fixture(scope="module")
def P():
    import __graft_entry__

    __graft_entry__.build()
    from piecewise_sparse_attention_gb300 import pisa

    pisa.load()
    return pisa


@pytest.mark.parametrize("grid,prefix", [((21, 30, 52), 0), ((1, 64, 64), 512), ((16, 64, 64), 0),
                                         ((3, 5, 7), 2), ((1, 1, 1), 0), ((2, 1, 300), 7),
                                         ((32, 64, 64), 0)])
def test_morton_permutation_parity(P, grid, prefix):
    st = P.new_status()
    perm = P.morton_permutation(grid, prefix, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    assert np.array_equal(perm.cpu().numpy(), oracle.morton_permutation(grid, prefix))


@pytest.mark.parametrize("dtype,n,heads,d", [(torch.bfloat16, 32760, 4, 128), (torch.float32, 777, 3, 64),
                                             (torch.bfloat16, 64, 1, 64), (torch.float32, 5000, 2, 128)])
def test_reorder_and_restore_bit_exact(P, dtype, n, heads, d):
    g = torch.Generator(device="cuda").manual_seed(n)
    x = torch.randn(n, heads, d, device="cuda", generator=g).to(dtype)
    perm = torch.randperm(n, device="cuda", generator=g).to(torch.int32)
    st = P.new_status()
    o = P.reorder_heads(x, perm, status=st)
    y = P.restore_heads(o, perm, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    xs = x.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).cpu().numpy()
    os_ = o.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).cpu().numpy()
    ps = perm.cpu().numpy()
    assert np.array_equal(os_, oracle.reorder_heads(xs, ps))
    assert torch.equal(y, x)


def test_reorder_reports_bad_permutation(P):
    x = torch.zeros(100, 2, 64, device="cuda")
    perm = torch.arange(100, device="cuda", dtype=torch.int32)
    perm[7] = -1
    perm[9] = 100
    st = P.new_status()
    P.reorder_heads(x, perm, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == P.ERR_DEVICE_CHECK


def check_route(got, qbar, kbar, scale, topk, band, n_sink, bias=None):
    return check_route_rows(got, qbar, kbar, scale, topk, band, bias=bias, n_sink=n_sink)[0]


def gpu_sets(idx, cnt):
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    return [[list(map(int, idx[h, i, : cnt[h, i]])) for i in range(idx.shape[1])]
            for h in range(idx.shape[0])]


@pytest.mark.parametrize("nb,d,topk,band,n_sink,cov", [(40, 128, 5, 1, 1, False), (300, 128, 17, 1, 8, False),
                                                        (64, 64, 10, 0, 3, True), (20, 128, 4, 1, 25, False),
                                                        (500, 128, 30, 2, 8, True), (7, 64, 2, 1, 0, False)])
def test_route_ex_sinks_parity(P, nb, d, topk, band, n_sink, cov):
    rng = np.random.default_rng(nb + n_sink)
    qbar = rng.standard_normal((2, nb, d)).astype(np.float32)
    kbar = rng.standard_normal((2, nb, d)).astype(np.float32)
    M = np.exp(rng.standard_normal((2, nb))).astype(np.float32) if cov else None
    idx, cnt = P.route_ex(torch.from_numpy(qbar).cuda(), torch.from_numpy(kbar).cuda(), 0.1, topk,
                          band, n_sink, mnorm=torch.from_numpy(M).cuda() if cov else None)
    got = gpu_sets(idx, cnt)
    for h in range(2):
        bias = oracle.covariance_bias(M[h].astype(np.float64), 1e-6) if cov else None
        check_route(got[h], qbar[h], kbar[h], 0.1, topk, band, n_sink, bias)


def test_flux_chain_with_reorder_and_text_sinks(P):
    """FLUX-like MMDiT layout: 512 text tokens then a 64 x 64 image grid, held
    token-major [n, H, d]. Morton-reorder the image tokens behind the text
    prefix, route with the 8 text blocks as sinks, run the forward, restore
    the token order; against the oracle doing the same on two heads."""
    wl = WORKLOADS["flux"]
    heads = [0, 5, wl.heads - 1]
    qs, ks, vs = zip(*(make_head(wl, h) for h in heads))
    tok = [np.ascontiguousarray(np.stack(a, axis=1)) for a in (qs, ks, vs)]  # [n, H, d]
    n_sink = wl.n_text // 64
    st = P.new_status()
    perm = P.morton_permutation(wl.grid, wl.n_text, status=st)
    tq, tk, tv = (P.reorder_heads(torch.from_numpy(a).cuda().bfloat16(), perm, status=st) for a in tok)
    qb, kb, _, _ = P.block_stats(tq, tk, tv, status=st)
    idx, cnt = P.route_ex(qb, kb, wl.scale, wl.topk, wl.band, n_sink, status=st)
    o = P.forward(tq, tk, tv, idx, cnt, wl.scale, out_dtype=torch.float32, status=st)
    y = P.restore_heads(o, perm, status=st).cpu().numpy()
    torch.cuda.synchronize()
    P.check_status(st)
    got = gpu_sets(idx, cnt)
    ps = oracle.morton_permutation(wl.grid, wl.n_text)
    for x in (0, 2):
        q, k, v = (oracle.reorder_heads(a, ps)[x] for a in tok)
        sto = oracle.block_stats(q, k, v, 64)
        sets = check_route(got[x], sto[0], sto[1], wl.scale, wl.topk, wl.band, n_sink)
        ref = oracle.forward(q, k, v, 64, wl.scale, sets, stats=sto)
        ref_tok = oracle.restore_heads(ref[None], ps)[:, 0]
        err = np.abs(y[:, x] - ref_tok).max()
        cos = (y[:, x] * ref_tok).sum(1) / (np.linalg.norm(y[:, x], axis=1) * np.linalg.norm(ref_tok, axis=1))
        assert err <= 2e-2 and cos.min() >= 0.9999, (err, cos.min())
