"""The one-call API, piecewise_sparse_attention(), with the widened options
(hybrid order, covariance routing, second-order mass and ranking bonus, sink
blocks): its output against the same entry points called one by one
(bit-identical: the same kernels), and the all-options chain against the
fp64 oracle."""

import math

import numpy as np
import pytest
import torch

import oracle
from route_check import check_route_rows
from piecewise_sparse_attention_gb300.workloads import small_case

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


def chained(P, q, k, v, topk, band, scale, variant, routing, norm, second_order, rank_bonus,
            n_sink, st):
    qb, kb, vs, _ = P.block_stats(q, k, v, status=st)
    hbar = P.global_first_order(k, v, kb, vs, status=st)
    M = P.block_heterogeneity(k, v, kb, hbar, norm=norm, status=st) if routing == "covariance" else None
    w = wrank = None
    if second_order:
        sp = P.second_order_spread(q, k, kb, scale, with_rank=rank_bonus, status=st)
        w, wrank = sp[0], (sp[3] if rank_bonus else None)
    if M is None and wrank is None and n_sink == 0:
        idx, cnt = P.route(qb, kb, scale, topk, band, status=st)
    else:
        idx, cnt = P.route_ex(qb, kb, scale, topk, band, n_sink, mnorm=M, bonus=wrank, status=st)
    if variant == "hybrid":
        return P.forward_hybrid(q, k, v, kb, vs, hbar, idx, cnt, scale, out_dtype=torch.float32,
                                status=st)
    if second_order:
        return P.forward_second_order(q, k, v, idx, cnt, w, scale, out_dtype=torch.float32, status=st)
    return P.forward(q, k, v, idx, cnt, scale, out_dtype=torch.float32, status=st)


@pytest.mark.parametrize("variant,routing,norm,second_order,rank_bonus,n_sink", [
    ("blockwise", "pooled", "spectral", False, False, 0),
    ("blockwise", "covariance", "spectral", False, False, 0),
    ("blockwise", "covariance", "frobenius", True, True, 2),
    ("blockwise", "pooled", "spectral", True, False, 1),
    ("hybrid", "pooled", "spectral", False, False, 0),
    ("hybrid", "covariance", "frobenius", False, False, 3)])
def test_one_call_matches_the_chained_calls(P, variant, routing, norm, second_order, rank_bonus,
                                            n_sink):
    q, k, v = small_case(2, 2000, 128, seed=77, dtype="bf16", spread=0.7)
    tq, tk, tv = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    s = 1 / math.sqrt(128)
    st = P.new_status()
    got = P.piecewise_sparse_attention(tq, tk, tv, topk=4, band=1, variant=variant, routing=routing,
                                       norm=norm, second_order=second_order, rank_bonus=rank_bonus,
                                       n_sink=n_sink, out_dtype=torch.float32, status=st)
    ref = chained(P, tq, tk, tv, 4, 1, s, variant, routing, norm, second_order, rank_bonus, n_sink, st)
    torch.cuda.synchronize()
    P.check_status(st)
    # bf16 with d = 128: Hbar is summed in a fixed order, so even the hybrid
    # output is the same bit for bit
    assert torch.equal(got, ref)


def test_one_call_rejects_bad_options(P):
    z = torch.zeros(1, 64, 64, device="cuda", dtype=torch.bfloat16)
    for kw in (dict(variant="dense"), dict(routing="softmax"), dict(variant="hybrid", second_order=True),
               dict(rank_bonus=True)):
        with pytest.raises(ValueError):
            P.piecewise_sparse_attention(z, z, z, topk=1, **kw)


@pytest.mark.parametrize("dtype,n,d", [("bf16", 3000, 128), ("f32", 1000, 64)])
def test_all_options_against_the_oracle(P, dtype, n, d):
    """Block-wise, covariance routing (Frobenius), second-order mass with its
    ranking bonus, 2 sink blocks: the route against the oracle's (near ties
    excepted), the output against the oracle on the GPU's route, taking the
    GPU's gate decision on spread entries within 1e-4 of ln n_j."""
    heads, topk, band, n_sink, eps = 2, 5, 1, 2, 1e-6
    q, k, v = small_case(heads, n, d, seed=5 + n, dtype=dtype, spread=0.9, mean_scale=1.2)
    tq, tk, tv = dev(q, dtype), dev(k, dtype), dev(v, dtype)
    s = 1 / math.sqrt(d)
    st = P.new_status()
    out = P.piecewise_sparse_attention(tq, tk, tv, topk=topk, band=band, routing="covariance",
                                       norm="frobenius", eps=eps, second_order=True, rank_bonus=True,
                                       n_sink=n_sink, out_dtype=torch.float32, status=st)
    # the same route and spread, for the comparison
    qb, kb, vs, _ = P.block_stats(tq, tk, tv, status=st)
    hbar = P.global_first_order(tk, tv, kb, vs, status=st)
    M = P.block_heterogeneity(tk, tv, kb, hbar, norm="frobenius", status=st)
    w, _, _, wrank = P.second_order_spread(tq, tk, kb, s, with_rank=True, status=st)
    idx, cnt = P.route_ex(qb, kb, s, topk, band, n_sink, mnorm=M, eps=eps, bonus=wrank, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    out, idx, cnt, w = out.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy(), w.cpu().double().numpy()
    nb = -(-n // 64)
    nj = np.array([min(64, n - 64 * j) for j in range(nb)])
    for h in range(heads):
        sto = oracle.block_stats(q[h], k[h], v[h], 64)
        H = sto[3]
        bias = oracle.covariance_bias(oracle.block_heterogeneity(H, oracle.global_first_order(H),
                                                                 "frobenius"), eps)
        spread = oracle.second_order_spread(q[h], k[h], 64, s)
        bonus = oracle.second_order_rank_bonus(spread, nj)
        got = [list(map(int, idx[h, i, :cnt[h, i]])) for i in range(nb)]
        sets, _ = check_route_rows(got, sto[0], sto[1], s, topk, band, bias=bias, n_sink=n_sink,
                                   bonus=bonus)
        gate = oracle.gate_second_order(spread, nj)
        near = np.abs(spread - np.log(nj.astype(np.float64))[None, :]) < NEAR
        gate[near] = np.where(w[h][near] == 0.0, 0.0, spread[near])
        ref = oracle.forward(q[h], k[h], v[h], 64, s, sets, stats=sto, spread=gate)
        got = np.asarray(out[h], np.float64)
        err = np.abs(got - ref).max()
        if dtype == "f32":
            assert err <= 1e-4, err
        else:
            cos = (got * ref).sum(1) / (np.linalg.norm(got, axis=1) * np.linalg.norm(ref, axis=1) + 1e-300)
            assert err <= 2e-2 and cos.min() >= 0.9999, (err, cos.min())


@pytest.mark.parametrize("options", [
    dict(variant="hybrid", routing="covariance", norm="frobenius", n_sink=1),
    dict(second_order=True, rank_bonus=True, n_sink=2)])
def test_host_pipeline_with_options(P, options):
    """piecewise_sparse_attention_host (pinned host buffers, tapered head
    groups) with the widened options against the one-call API on the device."""
    q, k, v = small_case(5, 1500, 128, seed=41, dtype="bf16", spread=0.8)
    host = [torch.from_numpy(a).to(torch.bfloat16).pin_memory() for a in (q, k, v)]
    out = torch.empty(5, 1500, 128, dtype=torch.bfloat16).pin_memory()
    st = P.new_status()
    P.piecewise_sparse_attention_host(*host, out, topk=3, band=1, chunks=3, taper=True,
                                      status=st, **options)
    ref = P.piecewise_sparse_attention(*(t.cuda() for t in host), topk=3, band=1,
                                       out_dtype=torch.bfloat16, status=st, **options)
    torch.cuda.synchronize()
    P.check_status(st)
    got = out.float()
    ref = ref.cpu().float()
    assert torch.equal(got, ref)


def test_host_pipeline_from_two_threads(P):
    """Two threads, each on its own current stream, run the host pipeline
    (whose device buffers are shared) on different inputs at the same time;
    both outputs equal the one-call API's."""
    import threading

    cases = [small_case(4, 1000, 128, seed=70 + t, dtype="bf16", spread=0.8) for t in range(2)]
    hosts = [[torch.from_numpy(a).to(torch.bfloat16).pin_memory() for a in c] for c in cases]
    outs = [torch.empty(4, 1000, 128, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    errors = []

    def work(t):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(5):
                    P.piecewise_sparse_attention_host(*hosts[t], outs[t], topk=3, band=1, chunks=3)
            s.synchronize()
        except Exception as e:  # reported below
            errors.append(e)

    th = [threading.Thread(target=work, args=(t,)) for t in range(2)]
    for x in th:
        x.start()
    for x in th:
        x.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for t in range(2):
        ref = P.piecewise_sparse_attention(*(a.cuda() for a in hosts[t]), topk=3, band=1,
                                           out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert torch.equal(outs[t], ref.cpu())


@pytest.mark.parametrize("heads,n,groups,taper,out_dtype", [
    (6, 4096, 3, True, torch.bfloat16), (5, 1000, 1, False, torch.float32),
    (7, 2048, 7, True, torch.bfloat16)])
def test_attention_host_c_entry_matches_python_pipeline(P, heads, n, groups, taper, out_dtype):
    """pisa_attention_host (copies, streams and events in C) gives the same
    bits as the Python host pipeline and as the three device calls."""
    d, topk, band = 128, 5, 1
    q, k, v = small_case(heads, n, d, seed=11, dtype="bf16", spread=0.7)
    hq, hk, hv = (torch.from_numpy(a).to(torch.bfloat16).pin_memory() for a in (q, k, v))
    st = P.new_status()
    out_c = torch.empty(heads, n, d, dtype=out_dtype).pin_memory()
    P.attention_host(hq, hk, hv, out_c, topk=topk, band=band, groups=groups, taper=taper,
                     status=st)
    out_py = torch.empty_like(out_c).pin_memory()
    P.piecewise_sparse_attention_host(hq, hk, hv, out_py, topk=topk, band=band, chunks=groups,
                                      taper=taper, status=st)
    tq, tk, tv = (t.cuda() for t in (hq, hk, hv))
    ref = P.piecewise_sparse_attention(tq, tk, tv, topk=topk, band=band, out_dtype=out_dtype,
                                       status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    assert torch.equal(out_c, out_py)
    assert torch.equal(out_c, ref.cpu())


def test_attention_host_follows_the_callers_stream(P):
    """Work already on the caller's stream (here: filling the inputs on the
    device and copying them back) comes before the call, and the caller's
    stream continues only after the downloads."""
    heads, n, d = 4, 2048, 128
    s = torch.cuda.Stream()
    hq, hk, hv = (torch.empty(heads, n, d, dtype=torch.bfloat16).pin_memory() for _ in range(3))
    out = torch.zeros(heads, n, d, dtype=torch.bfloat16).pin_memory()
    g = torch.Generator(device="cuda").manual_seed(5)
    with torch.cuda.stream(s):
        dev = [torch.randn(heads, n, d, device="cuda", generator=g).bfloat16() for _ in range(3)]
        for h, x in zip((hq, hk, hv), dev):
            h.copy_(x, non_blocking=True)
        P.attention_host(hq, hk, hv, out, topk=4, band=1, groups=4, taper=True, stream=s)
        check = out.cuda(non_blocking=True)
    s.synchronize()
    ref = P.piecewise_sparse_attention(*dev, topk=4, band=1, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(check, ref)
