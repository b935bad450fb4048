"""Seeded sweep over many small shapes: the block-wise forward, the hybrid
forward and the route of every case against the fp64 oracle. Shapes cover
n = 1 .. ~3000 (ragged tails, a single partial block), d = 64 and 128, bf16
and float32, band 0 .. 3 and top-k from 0 to beyond n_b (dense)."""

import math

import numpy as np
import pytest
import torch

import oracle
from route_check import check_route_rows
from piecewise_sparse_attention_gb300.workloads import small_case

pytestmark = pytest.mark.gpu



@pytest.fixture(scope="module")
def P():
    import __graft_entry__

    __graft_entry__.build()
    from piecewise_sparse_attention_gb300 import pisa

    pisa.load()
    return pisa


def cases(count=120, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for c in range(count):
        n = int(rng.choice([1, 7, 63, 64, 65, 127, 129, 200, 511, 777, 1024, 1500, 2049, 3000]))
        d = int(rng.choice([64, 128]))
        dtype = "bf16" if rng.random() < 0.7 else "f32"
        nb = -(-n // 64)
        band = int(rng.integers(0, 4))
        topk = int(rng.choice([0, 1, 2, max(1, nb // 8), nb, nb + 3]))
        heads = int(rng.integers(1, 4))
        spread = float(rng.choice([0.3, 0.8, 1.5]))
        out.append((c, n, d, dtype, band, topk, heads, spread))
    return out


def check_output(got, ref, dtype):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref).max()
    if dtype == "f32":
        assert err <= 1e-4, err
    else:
        cos = (got * ref).sum(1) / (np.linalg.norm(got, axis=1) * np.linalg.norm(ref, axis=1) + 1e-300)
        assert err <= 2e-2 and cos.min() >= 0.9999, (err, cos.min())


@pytest.mark.parametrize("c,n,d,dtype,band,topk,heads,spread", cases())
def test_sweep(P, c, n, d, dtype, band, topk, heads, spread):
    q, k, v = small_case(heads, n, d, seed=900 + c, dtype=dtype, spread=spread, mean_scale=1.0)
    conv = (lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(torch.bfloat16)) \
        if dtype == "bf16" else (lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().float())
    tq, tk, tv = conv(q), conv(k), conv(v)
    s = 1 / math.sqrt(d)
    st = P.new_status()
    qb, kb, vs, _ = P.block_stats(tq, tk, tv, status=st)
    hbar = P.global_first_order(tk, tv, kb, vs, status=st)
    idx, cnt = P.route(qb, kb, s, topk, band, status=st)
    out = P.forward(tq, tk, tv, idx, cnt, s, out_dtype=torch.float32, status=st)
    outh = P.forward_hybrid(tq, tk, tv, kb, vs, hbar, idx, cnt, s, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    out, outh = out.cpu().numpy(), outh.cpu().numpy()
    nb = -(-n // 64)
    for h in range(heads):
        sto = oracle.block_stats(q[h], k[h], v[h], 64)
        got = [list(map(int, idx[h, i, :cnt[h, i]])) for i in range(nb)]
        sets, _ = check_route_rows(got, sto[0], sto[1], s, topk, band)
        check_output(out[h], oracle.forward(q[h], k[h], v[h], 64, s, sets, stats=sto), dtype)
        check_output(outh[h], oracle.forward_hybrid(q[h], k[h], v[h], 64, s, sets, stats=sto), dtype)
