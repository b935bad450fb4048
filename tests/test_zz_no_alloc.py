"""pisa_forward_hybrid_static, the entry point for callers that cannot
allocate device memory (a plugin that is handed only its input and output
pointers, code whose device allocator belongs to another runtime, a component
that must not change the device footprint while it runs).

Checked through the C ABI:
* two calls in a row give the same bits as pisa_forward_hybrid (whose scratch
  the caller allocates): both run the same deterministic kernel on the same
  inputs, so any slip in the fixed array's layout would show;
* a size whose scratch fills the fixed array exactly runs, one block more is
  refused with an error message and nothing launched;
* the calls allocate nothing: the device's free memory is the same before and
  after them.

This file is collected last on purpose (the name sorts after every other
test file): the fixed array is shared by all calls, so a failure here should
not stop a first-failure run before the other tests have run."""

import ctypes
import math

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


def _scratch_bytes(heads, n, d):
    """What the hybrid tensor-core kernel keeps in the operand scratch: bf16
    hi and lo copies of kbar and Vhat ([heads, nb, d] each) and of Hbar
    ([heads, d, d])."""
    nb = -(-n // 64)
    return (4 * heads * nb * d + 2 * heads * d * d) * 2


def _workspace_bytes(heads, n, d):
    """The workspace of pisa_forward_hybrid: the operand scratch rounded up
    to 256 bytes, then the plan of the kernel's work (four int32 query block
    indices per 256 query rows and head), which the static entry point keeps
    in a second fixed array."""
    return -(-_scratch_bytes(heads, n, d) // 256) * 256 + heads * 4 * -(-n // 256) * 4


def _prepare(P, tq, tk, tv, topk):
    d = tq.shape[-1]
    s = 1 / math.sqrt(d)
    qb, kb, vs, _ = P.block_stats(tq, tk, tv)
    hbar = P.global_first_order(tk, tv, kb, vs)
    idx, cnt = P.route(qb, kb, s, topk, 1)
    return kb, vs, hbar, idx, cnt, s


def _small_inputs(heads, n, d, seed):
    q, k, v = small_case(heads, n, d, seed=seed, dtype="bf16", spread=0.6)
    return [torch.from_numpy(a).cuda().bfloat16() for a in (q, k, v)]


def _large_inputs(heads, n, d, seed):
    """Seeded inputs generated on the device (the exact-capacity case is too
    large to build on the host quickly): a per-block shared direction plus
    noise, so the route and both branches have work to do."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    nb = -(-n // 64)
    out = []
    for _ in range(3):
        base = torch.randn(heads, nb, 1, d, device="cuda", generator=g)
        x = base.expand(heads, nb, 64, d).reshape(heads, nb * 64, d)[:, :n]
        x = x + 0.5 * torch.randn(heads, n, d, device="cuda", generator=g)
        out.append((x * d ** -0.25).bfloat16().contiguous())
    return out


def _run_pair(P, tq, tk, tv, topk):
    """The workspace entry point once, then the static one twice in a row;
    returns (reference, [two static outputs], free bytes before and after the
    two static calls)."""
    kb, vs, hbar, idx, cnt, s = _prepare(P, tq, tk, tv, topk)
    st = P.new_status()
    ref = P.forward_hybrid(tq, tk, tv, kb, vs, hbar, idx, cnt, s, out_dtype=torch.float32,
                           status=st)
    outs = [torch.full_like(ref, float("nan")) for _ in range(2)]
    warm = torch.empty_like(ref)
    P.forward_hybrid_static(tq, tk, tv, kb, vs, hbar, idx, cnt, s, out=warm, status=st)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for o in outs:  # two calls in a row share the fixed scratch array
        P.forward_hybrid_static(tq, tk, tv, kb, vs, hbar, idx, cnt, s, out=o, status=st)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    P.check_status(st)
    return ref, outs, free0, free1


@pytest.mark.parametrize("heads,n,topk,seed", [(3, 4096, 11, 1), (2, 1000, 3, 2)])
def test_static_scratch_matches_workspace_entry_point(P, heads, n, topk, seed):
    tq, tk, tv = _small_inputs(heads, n, 128, seed)
    ref, outs, free0, free1 = _run_pair(P, tq, tk, tv, topk)
    for o in outs:
        assert torch.isfinite(o).all()
        assert torch.equal(o, ref)
    assert free1 == free0, "the static entry point changed the device's free memory"


def test_static_scratch_at_exact_capacity(P):
    L = P.load()
    cap = L.pisa_forward_hybrid_static_capacity()
    heads, n, d = 384, 4096, 128
    assert _scratch_bytes(heads, n, d) == cap
    assert L.pisa_forward_hybrid_workspace_size(P.BF16, heads, n, d) == _workspace_bytes(heads, n, d)
    tq, tk, tv = _large_inputs(heads, n, d, seed=7)
    ref, outs, free0, free1 = _run_pair(P, tq, tk, tv, topk=8)
    for o in outs:
        assert torch.isfinite(o).all()
        assert torch.equal(o, ref)
    assert free1 == free0


def test_static_scratch_rejects_sizes_beyond_its_array(P):
    L = P.load()
    cap = L.pisa_forward_hybrid_static_capacity()
    assert cap == 48 << 20
    # one key block beyond the exact-capacity case, and a far larger size;
    # the size check comes before anything is launched (pointers never read)
    fake = ctypes.c_void_p(0x10000)
    for heads, n in ((384, 4097), (64, 1 << 20)):
        assert _scratch_bytes(heads, n, 128) > cap
        rc = L.pisa_forward_hybrid_static(fake, fake, fake, 1, heads, n, 128, 64,
                                          ctypes.c_float(0.088), fake, fake, fake, fake, fake, 11,
                                          fake, 1, None, None)
        assert rc == P.ERR_UNSUPPORTED
        assert "scratch" in P.last_error()


def test_static_binding_refuses_what_it_would_have_to_copy(P):
    """The binding makes no hidden copies or allocations: a strided input or a
    wrong-sized output is refused before the call."""
    tq, tk, tv = _small_inputs(1, 256, 128, seed=3)
    kb, vs, hbar, idx, cnt, s = _prepare(P, tq, tk, tv, 1)
    out = torch.empty(1, 256, 128, device="cuda")
    with pytest.raises(ValueError):
        P.forward_hybrid_static(tq, tk, tv, kb, vs, hbar.transpose(1, 2), idx, cnt, s, out=out)
    with pytest.raises(ValueError):
        P.forward_hybrid_static(tq, tk, tv, kb, vs, hbar, idx, cnt, s, out=out[:, :255])
    with pytest.raises(TypeError):
        P.forward_hybrid_static(tq, tk, tv, kb, vs, hbar, idx, cnt, s,
                                out=torch.empty(1, 256, 128, device="cuda", dtype=torch.float16))
