"""pisa_forward_hybrid_static, the entry point for callers that cannot
allocate device memory: it must give the same output as pisa_forward_hybrid
(whose scratch buffer the caller allocates) on two calls in a row, through
the C ABI, and refuse sizes whose scratch exceeds its fixed array.

This file is collected last on purpose (the name sorts after every other
test file): the fixed array is shared by all calls, so a failure here should
not stop a first-failure run before the other tests have run."""

import ctypes
import math

import numpy as np
import pytest
import torch

from piecewise_sparse_attention_gb300.workloads import small_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    import __graft_entry__

    __graft_entry__.build()
    from piecewise_sparse_attention_gb300 import pisa

    pisa.load()
    return pisa


def _inputs(P, heads, n, d, topk, seed):
    q, k, v = small_case(heads, n, d, seed=seed, dtype="bf16", spread=0.6)
    tq, tk, tv = (torch.from_numpy(a).cuda().bfloat16() for a in (q, k, v))
    s = 1 / math.sqrt(d)
    qb, kb, vs, _ = P.block_stats(tq, tk, tv)
    hbar = P.global_first_order(tk, tv, kb, vs)
    idx, cnt = P.route(qb, kb, s, topk, 1)
    return tq, tk, tv, kb, vs, hbar, idx, cnt, s


def _close(got, ref):
    """The parity bar of the bf16 tests: max-abs 2e-2 and per-row cosine 0.9999."""
    got, ref = got.double().cpu().numpy(), ref.double().cpu().numpy()
    got, ref = got.reshape(-1, got.shape[-1]), ref.reshape(-1, ref.shape[-1])
    assert np.abs(got - ref).max() <= 2e-2
    cos = (got * ref).sum(1) / (np.linalg.norm(got, axis=1) * np.linalg.norm(ref, axis=1) + 1e-300)
    assert cos.min() >= 0.9999


@pytest.mark.parametrize("heads,n,topk,seed", [(3, 4096, 11, 1), (2, 1000, 3, 2)])
def test_static_scratch_matches_workspace_entry_point(P, heads, n, topk, seed):
    d = 128
    tq, tk, tv, kb, vs, hbar, idx, cnt, s = _inputs(P, heads, n, d, topk, seed)
    st = P.new_status()
    ref = P.forward_hybrid(tq, tk, tv, kb, vs, hbar, idx, cnt, s, out_dtype=torch.float32,
                           status=st)
    outs = []
    for _ in range(2):  # two calls in a row share the fixed scratch array
        o = torch.full_like(ref, float("nan"))
        P.forward_hybrid_static(tq, tk, tv, kb, vs, hbar, idx, cnt, s, out=o, status=st)
        outs.append(o)
    torch.cuda.synchronize()
    P.check_status(st)
    for o in outs:
        assert torch.isfinite(o).all()
        _close(o, ref)
    assert torch.equal(outs[0], outs[1])


def test_static_scratch_rejects_sizes_beyond_its_array(P):
    L = P.load()
    cap = L.pisa_forward_hybrid_static_capacity()
    assert cap == 48 << 20
    # 64 heads x 1M tokens would need far more scratch than the array holds;
    # the size check comes before anything is launched (pointers never read)
    fake = ctypes.c_void_p(0x10000)
    rc = L.pisa_forward_hybrid_static(fake, fake, fake, 1, 64, 1 << 20, 128, 64,
                                      ctypes.c_float(0.088), fake, fake, fake, fake, fake, 131,
                                      fake, 1, None, None)
    assert rc == P.ERR_UNSUPPORTED
    assert "scratch" in P.last_error()
