"""GPU parity: every call of the C ABI against the fp64 oracle on the same
seeded inputs.

Bars (from the method's accuracy targets):
* block statistics: means/sums within a few float32 ulps of the exact value;
  H within float32 (or bf16) storage precision;
* routing: block lists identical to the oracle's, except on rows where the
  oracle's k-th / (k+1)-th score gap is below 1e-5 (a near tie, where either
  choice is valid); such rows must still be a valid top-k within 1e-5;
* forward: max-abs error <= 1e-4 for float32 inputs; max-abs <= 2e-2 and
  per-row cosine >= 0.9999 for bf16 inputs. Where a near tie made the GPU
  route differ, the oracle output is evaluated on the GPU's route.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from piecewise_sparse_attention_gb300.workloads import WORKLOADS, make_head, small_case
from route_check import check_route_rows

pytestmark = pytest.mark.gpu



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


def check_route_head(got, qbar, kbar, scale, topk, band):
    """One head's GPU sets against the oracle (the shared near-tie rule);
    returns the sets to use for the forward comparison and the number of
    near-tie rows that differed."""
    return check_route_rows(got, qbar, kbar, scale, topk, band)


def check_output(got, ref, in_dtype):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref).max()
    if in_dtype == "f32":
        assert err <= 1e-4, err
    else:
        cos = (got * ref).sum(1) / (np.linalg.norm(got, axis=1) * np.linalg.norm(ref, axis=1) + 1e-300)
        assert err <= 2e-2, err
        assert cos.min() >= 0.9999, cos.min()
    return err


# ---------------------------------------------------------------------------
# tensor-core building blocks
# ---------------------------------------------------------------------------

def test_selftest_tensor_core_products(P):
    g = torch.Generator(device="cuda").manual_seed(0)
    a = torch.randn(128, 128, device="cuda", generator=g).bfloat16()
    b = torch.randn(128, 128, device="cuda", generator=g).bfloat16()
    bt = torch.randn(128, 128, device="cuda", generator=g).bfloat16()
    st = P.new_status()
    out = P.selftest_tc(a, b, bt, 0, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    ref1 = a.double() @ b.double().T
    ref2 = a.double() @ bt.double()
    ref3 = a.double().T @ bt.double()
    for got, ref in ((out[0], ref1), (out[1], ref2), (out[2], ref2), (out[3], ref3)):
        assert torch.allclose(got.double(), ref, rtol=1e-5, atol=1e-3), (got - ref).abs().max()


def test_selftest_bounded_wait_reports_timeout(P):
    z = torch.zeros(128, 128, device="cuda", dtype=torch.bfloat16)
    st = P.new_status()
    P.selftest_tc(z, z, z, 1, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == P.ERR_TIMEOUT
    # the context is still usable afterwards
    assert float(torch.ones(4, device="cuda").sum().item()) == 4.0


# ---------------------------------------------------------------------------
# block statistics
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,d,n", [("bf16", 128, 1000), ("bf16", 64, 64), ("f32", 64, 1000),
                                       ("f32", 128, 37), ("bf16", 128, 4096)])
def test_block_stats_parity(P, dtype, d, n):
    heads = 3
    q, k, v = small_case(heads, n, d, seed=n + d, dtype=dtype, spread=0.7, mean_scale=3.0)
    tq, tk, tv = dev(q, dtype), dev(k, dtype), dev(v, dtype)
    qb, kb, vs, H = P.block_stats(tq, tk, tv, with_h=True, h_dtype=torch.float32)
    _, _, _, Hb = P.block_stats(tq, tk, tv, with_h=True, h_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    for h in range(heads):
        oq, ok, ov, oH, nj = oracle.block_stats(q[h], k[h], v[h], 64)
        for got, ref in ((qb[h], oq), (kb[h], ok), (vs[h], ov)):
            got = got.cpu().double().numpy()
            # one float32 rounding of the exact value (plus a little for n_j != 2^k)
            assert np.all(np.abs(got - ref) <= 2.5e-7 * np.abs(ref) + 1e-30), np.abs(got - ref).max()
        gH = H[h].cpu().double().numpy()
        scaleH = np.abs(oH).max(axis=(1, 2), keepdims=True)
        assert np.abs(gH - oH).max() <= 1e-5 * scaleH.max()
        gHb = Hb[h].cpu().double().numpy()
        assert np.all(np.abs(gHb - oH) <= 2.0 ** -8 * np.abs(oH) + 1e-6 * scaleH)


@pytest.mark.parametrize("h_dtype", [torch.float32, torch.bfloat16])
def test_block_stats_h_paths_agree(P, h_dtype):
    """bf16 inputs with d = 128 form H_j on the tensor cores (centred on the kbar
    the same call writes) when kbar is requested, and on the CUDA cores when
    it is not: both results against each other and the oracle."""
    heads, n, d = 2, 777, 128
    q, k, v = small_case(heads, n, d, seed=31, dtype="bf16", spread=0.7, mean_scale=3.0)
    tq, tk, tv = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    nb = -(-n // 64)
    L = P.load()
    code = 0 if h_dtype == torch.float32 else 1
    outs = []
    for with_kbar in (True, False):
        qb = torch.empty(heads, nb, d, device="cuda")
        kb = torch.empty_like(qb) if with_kbar else None
        hm = torch.full((heads, nb, d, d), float("nan"), device="cuda", dtype=h_dtype)
        st = P.new_status()
        rc = L.pisa_block_stats(P._ptr(tq), P._ptr(tk), P._ptr(tv), P._dtype_code(tq.dtype), heads,
                                n, d, 64, P._ptr(qb), P._ptr(kb), None, P._ptr(hm), code,
                                P._ptr(st), P._stream())
        assert rc == 0, P.last_error()
        torch.cuda.synchronize()
        P.check_status(st)
        outs.append(hm.double().cpu().numpy())
    tol = 1e-5 if h_dtype == torch.float32 else 2.0 ** -7
    for h in range(heads):
        oH = oracle.block_stats(q[h], k[h], v[h], 64)[3]
        scale = np.abs(oH).max()
        for got in outs:
            assert np.all(np.isfinite(got[h]))
            assert np.abs(got[h] - oH).max() <= tol * scale
        assert np.abs(outs[0][h] - outs[1][h]).max() <= 2 * tol * scale


@pytest.mark.parametrize("dtype,d,n", [("bf16", 128, 1000), ("bf16", 64, 777), ("f32", 64, 1000),
                                       ("f32", 128, 37), ("bf16", 128, 64), ("bf16", 128, 4097)])
@pytest.mark.parametrize("want", ["q", "k", "v", "qk", "kv", "qkv"])
def test_block_means_parity(P, dtype, d, n, want):
    """The means / sums path (no H), which the forward's route reads: every
    subset of requested outputs (one, two or three tensors per launch), full
    and ragged last blocks, against the oracle's fp64 statistics, within one
    float32 rounding of the exact value. Outputs not requested stay untouched."""
    heads = 3
    q, k, v = small_case(heads, n, d, seed=7 * n + d + len(want), dtype=dtype, spread=0.7,
                         mean_scale=3.0)
    tq, tk, tv = dev(q, dtype), dev(k, dtype), dev(v, dtype)
    nb = -(-n // 64)
    outs = {c: torch.full((heads, nb, d), float("nan"), device="cuda") for c in "qkv"}
    req = {c: (outs[c] if c in want else None) for c in "qkv"}
    st = P.new_status()
    rc = P.load().pisa_block_stats(P._ptr(tq), P._ptr(tk), P._ptr(tv), P._dtype_code(tq.dtype),
                                   heads, n, d, 64, P._ptr(req["q"]), P._ptr(req["k"]),
                                   P._ptr(req["v"]), None, 0, P._ptr(st), P._stream())
    assert rc == 0, P.last_error()
    torch.cuda.synchronize()
    P.check_status(st)
    for h in range(heads):
        ref = dict(zip("qkv", oracle.block_stats(q[h], k[h], v[h], 64)[:3]))
        for c in "qkv":
            got = outs[c][h].cpu().double().numpy()
            if c not in want:
                assert np.isnan(got).all()
                continue
            assert np.all(np.abs(got - ref[c]) <= 2.5e-7 * np.abs(ref[c]) + 1e-30), \
                (c, np.abs(got - ref[c]).max())


@pytest.mark.parametrize("dtype,d,n,heads", [("bf16", 128, 1000, 3), ("bf16", 128, 4096, 2),
                                             ("bf16", 64, 777, 2), ("f32", 64, 1000, 2),
                                             ("f32", 128, 130, 1), ("bf16", 128, 32760, 2)])
def test_global_first_order_parity(P, dtype, d, n, heads):
    """Hbar = (1/nb) sum_j H_j against the oracle's per-block H_j."""
    q, k, v = small_case(heads, n, d, seed=3 * n + d, dtype=dtype, spread=0.8, mean_scale=2.0)
    tq, tk, tv = dev(q, dtype), dev(k, dtype), dev(v, dtype)
    st = P.new_status()
    _, kb, vs, _ = P.block_stats(tq, tk, tv, status=st)
    hbar = P.global_first_order(tk, tv, kb, vs, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    for h in range(heads):
        ref = oracle.global_first_order(oracle.block_stats(q[h], k[h], v[h], 64)[3])
        got = hbar[h].cpu().double().numpy()
        scale_ref = np.abs(ref).max()
        assert np.abs(got - ref).max() <= 2e-5 * scale_ref + 1e-6, (np.abs(got - ref).max(), scale_ref)


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def test_route_integer_scores_ties_exact(P):
    """Integer block means: exact scores with many ties; the GPU must take the
    lowest-index choice exactly like the oracle."""
    rng = np.random.default_rng(5)
    for nb, topk, band in [(40, 5, 1), (33, 0, 2), (64, 100, 1), (7, 3, 0), (1, 2, 1), (300, 17, 1)]:
        qbar = rng.integers(-2, 3, size=(2, nb, 128)).astype(np.float32)
        kbar = rng.integers(-2, 3, size=(2, nb, 128)).astype(np.float32)
        idx, cnt = P.route(torch.from_numpy(qbar).cuda(), torch.from_numpy(kbar).cuda(), 0.125,
                           topk, band)
        got = gpu_sets(idx, cnt)
        assert idx.shape[-1] == P.max_sel(nb, topk, band)
        pad = idx.cpu().numpy()
        for h in range(2):
            ora = oracle.route(qbar[h], kbar[h], 0.125, topk, band)
            assert got[h] == [list(map(int, s)) for s in ora], (nb, topk, band, h)
            for i in range(nb):
                assert np.all(pad[h, i, len(got[h][i]):] == -1)


def test_route_mass_ties_take_the_exact_fallback(P):
    """Many equal scores around the k-th one (more than the per-row re-scoring
    capacity): the exact fallback must still pick the lowest indices."""
    rng = np.random.default_rng(11)
    for nb, topk, band, d in [(300, 17, 1, 128), (1000, 100, 2, 128), (700, 40, 0, 64)]:
        qbar = rng.integers(-2, 3, size=(2, nb, d)).astype(np.float32)
        base = rng.integers(-2, 3, size=(2, 1, d)).astype(np.float32)
        kbar = np.repeat(base, nb, axis=1)
        kbar[:, ::7, 0] += 1.0  # two score levels per row, each shared by many blocks
        idx, cnt = P.route(torch.from_numpy(qbar).cuda(), torch.from_numpy(kbar).cuda(), 0.1,
                           topk, band)
        got = gpu_sets(idx, cnt)
        for h in range(2):
            ora = oracle.route(qbar[h], kbar[h], 0.1, topk, band)
            assert got[h] == [list(map(int, s)) for s in ora], (nb, topk, band, h)


def test_route_random_means_exact(P):
    """Random float means (no exact ties): identical to the oracle except at
    near-ties, at several block counts including a large one."""
    rng = np.random.default_rng(12)
    for nb, topk in [(64, 8), (513, 64), (2048, 128)]:
        qbar = (rng.standard_normal((2, nb, 128)) * 3).astype(np.float32)
        kbar = (rng.standard_normal((2, nb, 128)) * 3).astype(np.float32)
        idx, cnt = P.route(torch.from_numpy(qbar).cuda(), torch.from_numpy(kbar).cuda(), 0.088,
                           topk, 1)
        got = gpu_sets(idx, cnt)
        for h in range(2):
            check_route_head(got[h], qbar[h].astype(np.float64), kbar[h].astype(np.float64), 0.088,
                             topk, 1)


@pytest.mark.parametrize("n,d,topk,band", [(1000, 128, 3, 1), (4096, 128, 11, 1), (700, 64, 2, 0),
                                            (64, 128, 4, 1), (130, 128, 0, 1), (3000, 64, 50, 2)])
def test_route_parity_from_inputs(P, n, d, topk, band):
    heads = 2
    q, k, v = small_case(heads, n, d, seed=n * 7 + topk, dtype="bf16", spread=1.0)
    tq, tk, tv = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    s = 1 / math.sqrt(d)
    qb, kb, _, _ = P.block_stats(tq, tk, tv, with_vsum=False)
    idx, cnt = P.route(qb, kb, s, topk, band)
    got = gpu_sets(idx, cnt)
    for h in range(heads):
        oq, ok, _, _, _ = oracle.block_stats(q[h], k[h], v[h], 64)
        check_route_head(got[h], oq, ok, s, topk, band)


# ---------------------------------------------------------------------------
# forward
# ---------------------------------------------------------------------------

def run_path(P, q, k, v, dtype, scale, topk, band, out_dtype=torch.float32):
    tq, tk, tv = dev(q, dtype), dev(k, dtype), dev(v, dtype)
    st = P.new_status()
    qb, kb, _, _ = P.block_stats(tq, tk, tv, with_vsum=False, status=st)
    idx, cnt = P.route(qb, kb, scale, topk, band, status=st)
    out = P.forward(tq, tk, tv, idx, cnt, scale, out_dtype=out_dtype, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    return out, gpu_sets(idx, cnt)


@pytest.mark.parametrize("dtype,n,d,topk,band", [
    ("bf16", 1000, 128, 3, 1), ("bf16", 4096, 128, 11, 1), ("bf16", 777, 128, 2, 0),
    ("bf16", 64, 128, 0, 0), ("bf16", 200, 128, 50, 1), ("bf16", 1000, 64, 3, 1),
    ("bf16", 4096, 64, 11, 1), ("bf16", 333, 64, 2, 2), ("bf16", 50, 64, 1, 1),
    ("f32", 1000, 64, 4, 1), ("f32", 333, 128, 2, 2), ("f32", 50, 64, 1, 1)])
def test_forward_parity_small(P, dtype, n, d, topk, band):
    heads = 2
    q, k, v = small_case(heads, n, d, seed=n + 13 * topk, dtype=dtype, spread=0.6)
    s = 1 / math.sqrt(d)
    out, sets = run_path(P, q, k, v, dtype, s, topk, band)
    out = out.cpu().numpy()
    for h in range(heads):
        st = oracle.block_stats(q[h], k[h], v[h], 64)
        used, _ = check_route_head(sets[h], st[0], st[1], s, topk, band)
        ref = oracle.forward(q[h], k[h], v[h], 64, s, used, stats=st)
        check_output(out[h], ref, dtype)


def test_forward_density_one_is_dense_attention(P):
    """Every block exact: the GPU output is dense softmax attention."""
    n, d = 1000, 128
    q, k, v = small_case(2, n, d, seed=99, dtype="bf16")
    s = 1 / math.sqrt(d)
    out, _ = run_path(P, q, k, v, "bf16", s, 1000, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(a).double()[None] for a in (q, k, v)), scale=s)[0].numpy()
    for h in range(2):
        check_output(out[h].cpu().numpy(), ref[h], "bf16")


def test_forward_bf16_output(P):
    n, d = 1000, 128
    q, k, v = small_case(2, n, d, seed=5, dtype="bf16")
    s = 1 / math.sqrt(d)
    o32, _ = run_path(P, q, k, v, "bf16", s, 3, 1, out_dtype=torch.float32)
    o16, _ = run_path(P, q, k, v, "bf16", s, 3, 1, out_dtype=torch.bfloat16)
    assert torch.equal(o16, o32.bfloat16())


@pytest.mark.parametrize("name", ["tiny", "flux"])
def test_workload_full(P, name):
    wl = WORKLOADS[name]
    heads = list(range(wl.heads)) if name == "tiny" else [0, 7, wl.heads - 1]
    qs, ks, vs = zip(*(make_head(wl, h) for h in heads))
    q, k, v = np.stack(qs), np.stack(ks), np.stack(vs)
    out, sets = run_path(P, q, k, v, wl.dtype, wl.scale, wl.topk, wl.band)
    out = out.cpu().numpy()
    ties = 0
    for x in range(len(heads)):
        st = oracle.block_stats(q[x], k[x], v[x], wl.block)
        used, t = check_route_head(sets[x], st[0], st[1], wl.scale, wl.topk, wl.band)
        ties += t
        ref = oracle.forward(q[x], k[x], v[x], wl.block, wl.scale, used, stats=st)
        check_output(out[x], ref, wl.dtype)
    print(f"{name}: near-tie rows {ties}")


@pytest.mark.parametrize("name", ["wan", "hunyuan", "long"])
def test_workload_full_size_sampled(P, name):
    """Full launch shape of the workload; two heads hold the real workload
    (the rest is N(0,1) filler) and are checked on sampled query blocks
    (first, last/partial and four random ones) plus the whole route."""
    wl = WORKLOADS[name]
    H, n, d = wl.heads, wl.n, wl.d
    g = torch.Generator(device="cuda").manual_seed(1)
    tq, tk, tv = (torch.randn(H, n, d, device="cuda", generator=g).bfloat16() for _ in range(3))
    check = [0, H - 1]
    data = {}
    for h in check:
        q, k, v = make_head(wl, h)
        data[h] = (q, k, v)
        tq[h], tk[h], tv[h] = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    st = P.new_status()
    qb, kb, _, _ = P.block_stats(tq, tk, tv, with_vsum=False, status=st)
    idx, cnt = P.route(qb, kb, wl.scale, wl.topk, wl.band, status=st)
    out = P.forward(tq, tk, tv, idx, cnt, wl.scale, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    rng = np.random.default_rng(3)
    for h in check:
        q, k, v = data[h]
        sts = oracle.block_stats(q, k, v, wl.block)
        got = gpu_sets(idx[h:h + 1], cnt[h:h + 1])[0]
        used, ties = check_route_head(got, sts[0], sts[1], wl.scale, wl.topk, wl.band)
        blocks = sorted({0, wl.nb - 1, *rng.integers(1, wl.nb - 1, size=4).tolist()})
        ref = oracle.forward(q, k, v, wl.block, wl.scale, used, stats=sts, qblocks=blocks)
        o = out[h].cpu().numpy()
        for i in blocks:
            rows = slice(i * wl.block, min((i + 1) * wl.block, n))
            check_output(o[rows], ref[i], "bf16")


def test_python_chain_helper(P):
    q, k, v = small_case(2, 500, 128, seed=8, dtype="bf16")
    tq, tk, tv = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    o = P.piecewise_sparse_attention(tq, tk, tv, topk=2, band=1, out_dtype=torch.float32)
    s = 1 / math.sqrt(128)
    qb, kb, _, _ = P.block_stats(tq, tk, tv)
    idx, cnt = P.route(qb, kb, s, 2, 1)
    o2 = P.forward(tq, tk, tv, idx, cnt, s, out_dtype=torch.float32)
    assert torch.equal(o, o2)


def test_bad_route_entry_is_reported(P):
    q, k, v = small_case(1, 256, 128, seed=2, dtype="bf16")
    tq, tk, tv = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    idx = torch.tensor([[[0, 1, 9], [0, 1, 2], [1, 2, 3], [2, 3, -1]]], dtype=torch.int32,
                       device="cuda")
    cnt = torch.tensor([[3, 3, 3, 2]], dtype=torch.int32, device="cuda")
    st = P.new_status()
    out = P.forward(tq, tk, tv, idx, cnt, 0.088, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == P.ERR_DEVICE_CHECK
    assert torch.isfinite(out).all()


# ---------------------------------------------------------------------------
# hybrid-order forward (global Hbar)
# ---------------------------------------------------------------------------

def run_hybrid(P, q, k, v, dtype, scale, topk, band, out_dtype=torch.float32):
    tq, tk, tv = dev(q, dtype), dev(k, dtype), dev(v, dtype)
    st = P.new_status()
    qb, kb, vs, _ = P.block_stats(tq, tk, tv, status=st)
    hbar = P.global_first_order(tk, tv, kb, vs, status=st)
    idx, cnt = P.route(qb, kb, scale, topk, band, status=st)
    out = P.forward_hybrid(tq, tk, tv, kb, vs, hbar, idx, cnt, scale, out_dtype=out_dtype,
                           status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    return out, gpu_sets(idx, cnt)


@pytest.mark.parametrize("dtype,n,d,topk,band", [
    ("bf16", 1000, 128, 3, 1), ("bf16", 4096, 128, 11, 1), ("bf16", 777, 128, 2, 0),
    ("bf16", 64, 128, 0, 0), ("bf16", 200, 128, 50, 1), ("bf16", 1000, 64, 3, 1),
    ("bf16", 4096, 64, 11, 1), ("bf16", 130, 64, 0, 0),
    ("f32", 1000, 64, 4, 1), ("f32", 333, 128, 2, 2), ("f32", 50, 64, 1, 1)])
def test_forward_hybrid_parity_small(P, dtype, n, d, topk, band):
    heads = 2
    q, k, v = small_case(heads, n, d, seed=n + 17 * topk, dtype=dtype, spread=0.6)
    s = 1 / math.sqrt(d)
    out, sets = run_hybrid(P, q, k, v, dtype, s, topk, band)
    out = out.cpu().numpy()
    for h in range(heads):
        st = oracle.block_stats(q[h], k[h], v[h], 64)
        used, _ = check_route_head(sets[h], st[0], st[1], s, topk, band)
        ref = oracle.forward_hybrid(q[h], k[h], v[h], 64, s, used, stats=st)
        check_output(out[h], ref, dtype)


@pytest.mark.parametrize("name", ["tiny", "flux", "wan", "hunyuan", "long"])
def test_forward_hybrid_workloads(P, name):
    wl = WORKLOADS[name]
    heads = list(range(wl.heads)) if name == "tiny" else [0, wl.heads - 1]
    qs, ks, vs = zip(*(make_head(wl, h) for h in heads))
    q, k, v = np.stack(qs), np.stack(ks), np.stack(vs)
    out, sets = run_hybrid(P, q, k, v, wl.dtype, wl.scale, wl.topk, wl.band)
    out = out.cpu().numpy()
    rng = np.random.default_rng(4)
    for x in range(len(heads)):
        st = oracle.block_stats(q[x], k[x], v[x], wl.block)
        used, _ = check_route_head(sets[x], st[0], st[1], wl.scale, wl.topk, wl.band)
        blocks = None if wl.nb <= 72 else sorted({0, wl.nb - 1, *rng.integers(1, wl.nb - 1, 6).tolist()})
        ref = oracle.forward_hybrid(q[x], k[x], v[x], wl.block, wl.scale, used, stats=st,
                                    qblocks=blocks)
        if blocks is None:
            check_output(out[x], ref, wl.dtype)
        else:
            for i in blocks:
                rows = slice(i * wl.block, min((i + 1) * wl.block, wl.n))
                check_output(out[x][rows], ref[i], wl.dtype)


# ---------------------------------------------------------------------------
# host-buffer pipeline of the public API
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("chunks", [1, 3, 4])
def test_host_pipeline_matches_device_path(P, chunks):
    """piecewise_sparse_attention_host (head groups, overlapped copies) gives
    the same bits as the device-buffer call: every kernel is deterministic per
    head and the grouping only changes which launch a head is in."""
    wl = WORKLOADS["flux"]
    heads = list(range(7))
    qs, ks, vs = zip(*(make_head(wl, h) for h in heads))
    host = [torch.from_numpy(np.stack(a)).bfloat16().pin_memory() for a in (qs, ks, vs)]
    ref = P.piecewise_sparse_attention(*(t.cuda() for t in host), topk=wl.topk, band=wl.band,
                                       scale=wl.scale, out_dtype=torch.bfloat16)
    out = torch.empty_like(host[0]).pin_memory()
    st = P.new_status()
    P.piecewise_sparse_attention_host(*host, out, topk=wl.topk, band=wl.band, scale=wl.scale,
                                      chunks=chunks, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    assert torch.equal(out, ref.cpu())


def test_forward_head_dim_64_at_a_video_length(P):
    """bf16 with d = 64 on the tensor-core path at a Wan-like length
    (32760 tokens, a partial last block), sampled query blocks."""
    heads, n, d, topk, band = 2, 32760, 64, 64, 1
    q, k, v = small_case(heads, n, d, seed=64, dtype="bf16", spread=0.6)
    s = 1 / math.sqrt(d)
    tq, tk, tv = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    st = P.new_status()
    qb, kb, _, _ = P.block_stats(tq, tk, tv, status=st)
    idx, cnt = P.route(qb, kb, s, topk, band, status=st)
    out = P.forward(tq, tk, tv, idx, cnt, s, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    out = out.cpu().numpy()
    sets_all = gpu_sets(idx, cnt)
    nb = -(-n // 64)
    rng = np.random.default_rng(3)
    blocks = sorted({0, nb - 1, *rng.integers(1, nb - 1, 6).tolist()})
    for h in range(heads):
        stx = oracle.block_stats(q[h], k[h], v[h], 64)
        used, _ = check_route_head(sets_all[h], stx[0], stx[1], s, topk, band)
        ref = oracle.forward(q[h], k[h], v[h], 64, s, used, stats=stx, qblocks=blocks)
        for i in blocks:
            rows = slice(i * 64, min((i + 1) * 64, n))
            check_output(out[h][rows], ref[i], "bf16")


def test_forward_hybrid_head_dim_64_at_a_video_length(P):
    """Hybrid order, bf16 with d = 64 on the tensor-core path at a Wan-like
    length (32760 tokens, a partial last block), sampled query blocks."""
    heads, n, d, topk, band = 2, 32760, 64, 64, 1
    q, k, v = small_case(heads, n, d, seed=65, dtype="bf16", spread=0.6)
    s = 1 / math.sqrt(d)
    out, sets = run_hybrid(P, q, k, v, "bf16", s, topk, band)
    out = out.cpu().numpy()
    nb = -(-n // 64)
    rng = np.random.default_rng(5)
    blocks = sorted({0, nb - 1, *rng.integers(1, nb - 1, 6).tolist()})
    for h in range(heads):
        st = oracle.block_stats(q[h], k[h], v[h], 64)
        used, _ = check_route_head(sets[h], st[0], st[1], s, topk, band)
        ref = oracle.forward_hybrid(q[h], k[h], v[h], 64, s, used, stats=st, qblocks=blocks)
        for i in blocks:
            rows = slice(i * 64, min((i + 1) * 64, n))
            check_output(out[h][rows], ref[i], "bf16")


def test_forward_offsets_past_2_31_elements(P):
    """136 heads x 131072 tokens x 128: the last head starts at element
    2.28e9 > 2^31, so every index of the stats, route, block-wise and hybrid
    kernels must be 64-bit where it has to be. N(0,1) filler everywhere
    (generated on the device); heads 0 and 135 hold seeded cases and are
    checked on sampled query blocks, the route in full."""
    H, n, d, topk, band = 136, 131072, 128, 128, 1
    s = 1 / math.sqrt(d)
    g = torch.Generator(device="cuda").manual_seed(2)
    tq, tk, tv = (torch.randn(H, n, d, device="cuda", generator=g, dtype=torch.bfloat16)
                  for _ in range(3))
    check = [0, H - 1]
    data = {}
    for i, h in enumerate(check):
        q, k, v = small_case(1, n, d, seed=31 + i, dtype="bf16", spread=0.6)
        data[h] = (q[0], k[0], v[0])
        tq[h], tk[h], tv[h] = dev(q[0], "bf16"), dev(k[0], "bf16"), dev(v[0], "bf16")
    st = P.new_status()
    qb, kb, vs, _ = P.block_stats(tq, tk, tv, status=st)
    hbar = P.global_first_order(tk, tv, kb, vs, status=st)
    idx, cnt = P.route(qb, kb, s, topk, band, status=st)
    sel = torch.tensor(check, device="cuda")
    sets = gpu_sets(idx[sel], cnt[sel])
    nb = -(-n // 64)
    rng = np.random.default_rng(9)
    blocks = sorted({0, nb - 1, *rng.integers(1, nb - 1, 3).tolist()})
    rows = torch.cat([torch.arange(i * 64, min((i + 1) * 64, n)) for i in blocks]).cuda()
    out = P.forward(tq, tk, tv, idx, cnt, s, out_dtype=torch.float32, status=st)
    got_fwd = out[sel][:, rows].cpu().numpy()
    del out
    out = P.forward_hybrid(tq, tk, tv, kb, vs, hbar, idx, cnt, s, out_dtype=torch.float32, status=st)
    got_hyb = out[sel][:, rows].cpu().numpy()
    del out
    torch.cuda.synchronize()
    P.check_status(st)
    for x, h in enumerate(check):
        q, k, v = data[h]
        stx = oracle.block_stats(q, k, v, 64)
        used, _ = check_route_head(sets[x], stx[0], stx[1], s, topk, band)
        ref = oracle.forward(q, k, v, 64, s, used, stats=stx, qblocks=blocks)
        refh = oracle.forward_hybrid(q, k, v, 64, s, used, stats=stx, qblocks=blocks)
        r0 = 0
        for i in blocks:
            m = min((i + 1) * 64, n) - i * 64
            check_output(got_fwd[x][r0:r0 + m], ref[i], "bf16")
            check_output(got_hyb[x][r0:r0 + m], refh[i], "bf16")
            r0 += m


def test_the_largest_head_count(P):
    """65535 heads (the grid.y limit of the per-head launches) x 64 tokens x 64,
    bf16: stats, route, block-wise and hybrid forward, both heterogeneity norms
    and the second-order spread launch and agree with the oracle on the first,
    a middle and the last head."""
    H, n, d, topk, band = 65535, 64, 64, 1, 1
    s = 1 / math.sqrt(d)
    g = torch.Generator(device="cuda").manual_seed(3)
    tq, tk, tv = (torch.randn(H, n, d, device="cuda", generator=g, dtype=torch.bfloat16)
                  for _ in range(3))
    check = [0, H // 2, H - 1]
    st = P.new_status()
    qb, kb, vs, _ = P.block_stats(tq, tk, tv, status=st)
    hbar = P.global_first_order(tk, tv, kb, vs, status=st)
    idx, cnt = P.route(qb, kb, s, topk, band, status=st)
    out = P.forward(tq, tk, tv, idx, cnt, s, out_dtype=torch.float32, status=st)
    outh = P.forward_hybrid(tq, tk, tv, kb, vs, hbar, idx, cnt, s, out_dtype=torch.float32, status=st)
    mf = P.block_heterogeneity(tk, tv, kb, hbar, norm="frobenius", status=st)
    ms = P.block_heterogeneity(tk, tv, kb, hbar, norm="spectral", status=st)
    w, _, _ = P.second_order_spread(tq, tk, kb, s, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    sel = torch.tensor(check, device="cuda")
    q, k, v = (t[sel].float().cpu().numpy() for t in (tq, tk, tv))
    out, outh = out[sel].cpu().numpy(), outh[sel].cpu().numpy()
    mf, ms, w = mf[sel].cpu().double().numpy(), ms[sel].cpu().double().numpy(), w[sel].cpu().numpy()
    for x in range(len(check)):
        sto = oracle.block_stats(q[x], k[x], v[x], 64)
        sets = [np.array([0], dtype=np.int64)]
        check_output(out[x], oracle.forward(q[x], k[x], v[x], 64, s, sets, stats=sto), "bf16")
        check_output(outh[x], oracle.forward_hybrid(q[x], k[x], v[x], 64, s, sets, stats=sto), "bf16")
        # one block: Hbar = H_0, so M_0 = 0 up to the float32 rounding of H_0
        top = np.sqrt((sto[3] ** 2).sum())
        assert mf[x][0] <= 1e-5 * top and ms[x][0] <= 1e-5 * top, (mf[x], ms[x], top)
        ref_w = oracle.second_order_spread(q[x], k[x], 64, s)
        gate = oracle.gate_second_order(ref_w, np.array([64]))
        assert abs(w[x][0, 0] - gate[0, 0]) <= 1e-4 * max(1.0, abs(gate[0, 0])) or \
            abs(ref_w[0, 0] - math.log(64)) < 1e-4, (w[x], ref_w)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 128), ("f32", 64)])
def test_global_first_order_is_deterministic(P, dtype, d):
    """The cluster reduction sums the partials of a head in a fixed order, so
    repeated calls give the same Hbar bit for bit (tensor-core and CUDA-core
    kernels alike)."""
    q, k, v = small_case(3, 5000, d, seed=8, dtype=dtype, spread=0.8, mean_scale=2.0)
    tk, tv = dev(k, dtype), dev(v, dtype)
    st = P.new_status()
    _, kb, vs, _ = P.block_stats(dev(q, dtype), tk, tv, status=st)
    first = P.global_first_order(tk, tv, kb, vs, status=st)
    for _ in range(5):
        again = P.global_first_order(tk, tv, kb, vs, status=st)
        torch.cuda.synchronize()
        assert torch.equal(first, again)
    P.check_status(st)
