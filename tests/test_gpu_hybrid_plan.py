"""The plan of the hybrid tensor-core kernel, read back from the workspace of
pisa_forward_hybrid after a call.

The plan decides which two query blocks share a 128-row query tile and which
two tiles share a CTA; it never changes which keys a row attends to (the
parity tests check the outputs). Here it is checked against its definition,
recomputed on the host from the route's critical sets:
* every query block of a head appears exactly once (the rest of the slots
  hold nb, "no block");
* the tiles are the greedy matching by overlap |S_a & S_b| over the pairs
  whose block indices differ by at most the window W (largest overlap first,
  then lower indices), the blocks it leaves unmatched paired in index order
  and an odd one out alone;
* the tiles run in order of decreasing exact tiles ceil(|S_a | S_b| / 2),
  lower first block first among equal ones, two per CTA.
"""

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


def _window(nb):
    """The matching window the library picks for nb blocks (0: neighbours)."""
    nw = 8 if nb <= 256 else 16 if nb <= 512 else 32 if nb <= 1024 else 0
    if nw == 0:
        return 0
    nt = (nb + 1) // 2
    p2 = 1
    while p2 < nt:
        p2 <<= 1
    for w in (128, 64, 32, 16):
        if (p2 + 2 * nt) * 4 + 3 * nb * 4 + nb * (nw + 4) * 4 + nb * w <= 220 * 1024:
            return w
    return 0


def _expected_tiles(sets, nb, W):
    if W == 0:
        return [(2 * t, 2 * t + 1 if 2 * t + 1 < nb else nb) for t in range((nb + 1) // 2)]
    edges = sorted((-min(len(sets[a] & sets[b]), 255), a, b)
                   for a in range(nb) for b in range(a + 1, min(nb, a + W + 1)))
    mate = [-1] * nb
    for _, a, b in edges:
        if mate[a] < 0 and mate[b] < 0:
            mate[a], mate[b] = b, a
    rest = [i for i in range(nb) if mate[i] < 0]
    for p in range(0, len(rest) - 1, 2):
        mate[rest[p]], mate[rest[p + 1]] = rest[p + 1], rest[p]
    if len(rest) % 2:
        mate[rest[-1]] = nb
    return [(i, mate[i]) for i in range(nb) if mate[i] > i]


@pytest.mark.parametrize("heads,nb,topk,seed", [(2, 37, 5, 1), (2, 300, 12, 2), (1, 8, 2, 3)])
def test_hybrid_plan_matches_its_definition(P, heads, nb, topk, seed):
    n, d = nb * 64 - 17, 128  # a partial last block
    q, k, v = small_case(heads, n, d, seed=seed, dtype="bf16", spread=0.6)
    tq, tk, tv = [torch.from_numpy(a).cuda().bfloat16() for a in (q, k, v)]
    s = 1 / math.sqrt(d)
    qb, kb, vs, _ = P.block_stats(tq, tk, tv)
    hbar = P.global_first_order(tk, tv, kb, vs)
    idx, cnt = P.route(qb, kb, s, topk, 1)
    L = P.load()
    nbytes = L.pisa_forward_hybrid_workspace_size(P.BF16, heads, n, d)
    ws = torch.zeros(nbytes, device="cuda", dtype=torch.uint8)
    P.forward_hybrid(tq, tk, tv, kb, vs, hbar, idx, cnt, s, workspace=ws)
    torch.cuda.synchronize()

    n_ctas = -(-n // 256)
    plan_off = -(-((4 * heads * nb * d + 2 * heads * d * d) * 2) // 256) * 256
    assert nbytes == plan_off + heads * 4 * n_ctas * 4
    plan = ws[plan_off:].cpu().numpy().view(np.int32).reshape(heads, n_ctas, 4)
    idx_h, cnt_h = idx.cpu().numpy(), cnt.cpu().numpy()
    W = _window(nb)
    for h in range(heads):
        sets = [set(idx_h[h, i, : cnt_h[h, i]].tolist()) for i in range(nb)]
        flat = plan[h].reshape(-1)
        assert sorted(flat[flat < nb].tolist()) == list(range(nb))
        assert (flat[flat >= nb] == nb).all()
        tiles = [(int(a), int(b)) for a, b in plan[h].reshape(-1, 2) if a < nb]
        assert sorted(tiles) == _expected_tiles(sets, nb, W)

        def te(t):
            return (len(sets[t[0]] | (sets[t[1]] if t[1] < nb else set())) + 1) // 2

        assert tiles == sorted(tiles, key=lambda t: (-te(t), t[0]))
        # the odd tile out, if any, is the last one and shares its CTA with nothing
        assert all(a == nb for a in plan[h].reshape(-1, 2)[len(tiles):, 0])
