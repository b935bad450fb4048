"""Comparison of a GPU route with the oracle's, shared by the GPU tests.

Routing is integer output decided by floating-point scores, so the two sides
must agree exactly except where the choice itself is not unique: on a row whose
oracle margin (the k-th minus the (k+1)-th ranked free score, the free blocks
being those outside the band and the sinks) is below 1e-5 in logit units, any
selection that is a valid top-k within that tolerance is accepted. The
selection rule is Figure 4 "Prepare Phase" / Algorithm 1 step 2 of the PISA
paper (top-k on s * qbar_i . kbar_j, with the Section 3.3 Eq. 11 bias when
given), the band and the sinks follow the Piecewise-Taylor-Attention README
("Knobs").
"""

import numpy as np

import oracle

GAP = 1e-5


def check_route_rows(got, qbar, kbar, scale, topk, band, bias=None, n_sink=0, bonus=None,
                     rows=None):
    """Checks the GPU sets ``got`` (one list of block indices per row of
    ``rows``, every query block when None) against the oracle.

    A row equal to the oracle's passes. A row that differs must have an oracle
    margin below GAP and must still be a valid selection: ascending, without
    repeats, holding every forced block (band and sinks) plus exactly
    min(topk, #free) free blocks, each picked score >= T - GAP and each
    unpicked free score <= T + GAP, T being the k-th ranked free score.
    Returns (the sets to evaluate the oracle's forward on, as int64 arrays;
    the number of near-tie rows that differed)."""
    nb = np.asarray(kbar).shape[0]
    want = list(range(nb)) if rows is None else list(rows)
    assert len(got) == len(want), (len(got), len(want))
    kw = dict(bias=bias, n_sink=n_sink, bonus=bonus, rows=want)
    ora = oracle.route(qbar, kbar, scale, topk, band, **kw)
    gaps = oracle.route_gaps(qbar, kbar, scale, topk, band, **kw)
    bon = None if bonus is None else np.asarray(bonus, np.float64)[want]
    r = oracle.route_scores(np.asarray(qbar, np.float64)[want], kbar, scale, bias, bon)
    used, ties = [], 0
    for a, i in enumerate(want):
        g = [int(x) for x in got[a]]
        o = [int(x) for x in ora[a]]
        if g != o:
            assert gaps[a] < GAP, f"row {i}: {g} != {o} with margin {gaps[a]:.3e}"
            ties += 1
            forced = {j for j in range(nb) if abs(i - j) <= band or j < n_sink}
            free = [j for j in range(nb) if j not in forced]
            take = min(topk, len(free))
            gs = set(g)
            assert g == sorted(g) and len(gs) == len(g), (i, g)
            assert forced <= gs and len(gs) == len(forced) + take, (i, g)
            assert all(0 <= j < nb for j in g), (i, g)
            if take:
                T = np.sort(r[a, free])[::-1][take - 1]
                assert all(r[a, j] >= T - GAP for j in gs - forced), (i, g, T)
                assert all(r[a, j] <= T + GAP for j in free if j not in gs), (i, g, T)
        used.append(np.array(g, dtype=np.int64))
    return used, ties
