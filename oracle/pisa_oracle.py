"""fp64 CPU reference ("oracle") for piecewise sparse attention (PISA).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The product path (the
CUDA library and its Python binding) never imports, links or executes it, and
this module imports nothing from the product package.

Everything below is plain NumPy in float64, one head at a time, following
"PISA: Piecewise Sparse Attention Is Wiser for Efficient Diffusion
Transformers" in the order the paper states the method:

* block partition and block statistics (Section 3.2 "Formulation";
  Appendix C "Notation"): query/key block means, value block sums and the
  block-wise first-order matrix H_j = sum_n (k_{j,n} - kbar_j)^T v_{j,n};
* block routing (Section 3.4, Figure 4 "Prepare Phase", Algorithm 1 step 2):
  pooled score s * qbar_i . kbar_j, top-k per query block, plus the +-1
  diagonal band kept exact (Piecewise-Taylor-Attention README, "Knobs":
  band=b keeps |i-j| <= b exact);
* the piecewise forward (Section 3.2, Eq. (3)-(6)): exact softmax terms for
  the selected blocks, and for every other block the zeroth-order mass
  n_j * exp(q'.kbar_j) in the denominator and exp(q'.kbar_j) (Vhat_j + q' H_j)
  in the numerator, all under one shared denominator.

Readings where the text is silent or ambiguous (each also listed in the design
notes of the repository):

* q' = s * q with s = 1/sqrt(d) by default, applied everywhere including the
  first-order term (Eq. (3)-(6) omit the scale; Appendix C puts 1/sqrt(d)
  inside alpha_{t,j}).
* H_j is centred on the block's own centroid (Appendix C, Eq. (6)), not the
  global centroid of Section 3.3.
* A partial last block of n_j < B tokens uses means over n_j tokens and mass
  n_j * alpha.
* Top-k is taken over the blocks outside the band; ties go to the lower block
  index; the band is added on top (|S_i| = k + |band(i)| away from the edges).
* The shift m used for numerical safety is the row maximum over every exact
  logit and every centroid logit (Figure 3 "Safe-Exp"); the result does not
  depend on it mathematically.
* Hybrid variant (Section 3.3 Eq. 7-10, Algorithm 1 Phase 3): the global
  first-order statistic is the mean of the block-centred H_j over all n_b
  blocks (Appendix C "Notation": Hbar = (1/N) sum_j H_j), query independent;
  the first-order numerator term is (sum_{j in U_i} alpha_tj) q' Hbar (Eq. 10),
  with the same block masses n_j alpha_tj in the denominator as Eq. 3.
  Algorithm 1's "L^{-1}" factor is read as the 1/n_b inside Hbar.
* Covariance-aware routing (Section 3.3 Eq. 11, Appendix D Eq. 14): the
  pooled score of key block j gains log(M_j + eps), M_j = ||H_j - Hbar|| with
  the same Hbar as the hybrid variant; Section 3.3 writes the spectral norm
  (the default here), the Piecewise-Taylor-Attention README uses the Frobenius
  norm (selectable). eps is not given on the pages; it is an argument.
* Second-order block mass (Piecewise-Taylor-Attention README): the spread
  w_ij uses the population variance (1/n_j) of each key channel of block j and
  the mean of the squared queries of query block i, with the scale entering
  squared (the expansion is in q' = s q); the gate compares w_ij with ln(n_j);
  w enters the logit of the approximated block, so both the mass and the
  Taylor numerator carry exp(w) (the README's "virtual-token logits").
* Second-order ranking bonus: the README's router adds min(w_ij, ln n_j) to
  the pooled score (clamped, not gated), with the same ungated w.
* Sink blocks (the README's n_sink_blocks): the first n_sink key blocks are
  forced into every S_i on top of the band; top-k is taken over the rest.
* Morton reorder: t is the most significant coordinate in every bit triple,
  then y, then x; a text prefix keeps its place in front of the grid tokens.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "n_blocks",
    "block_rows",
    "block_stats",
    "route_scores",
    "route",
    "route_gaps",
    "block_heterogeneity",
    "morton_permutation",
    "reorder_heads",
    "restore_heads",
    "covariance_bias",
    "forward",
    "forward_head",
    "global_first_order",
    "second_order_spread",
    "gate_second_order",
    "second_order_rank_bonus",
    "forward_hybrid",
]


def morton_permutation(grid, n_prefix: int = 0):
    """Token order of the Morton (Z-order) reorder of the Piecewise-Taylor-
    Attention README ("Morton tile reorder + fused gather"): the T x Y x X grid
    tokens (raster index (t Y + y) X + x) sorted by the code that interleaves
    the bits of t, y, x, bit b of t at position 3b + 2, of y at 3b + 1, of x at
    3b, over the power-of-two box that holds the grid; ``n_prefix`` leading
    tokens (a text prefix) keep their places in front. perm[p] = source index
    of the token at position p."""
    T, Y, X = grid
    bits = max(int(math.ceil(math.log2(max(T, Y, X, 2)))), 1)
    codes = []
    for t in range(T):
        for y in range(Y):
            for x in range(X):
                c = 0
                for b in range(bits):
                    c |= ((t >> b) & 1) << (3 * b + 2)
                    c |= ((y >> b) & 1) << (3 * b + 1)
                    c |= ((x >> b) & 1) << (3 * b)
                codes.append(c)
    order = np.argsort(np.array(codes, dtype=np.int64), kind="stable")
    return np.concatenate([np.arange(n_prefix), n_prefix + order]).astype(np.int64)


def reorder_heads(x, perm):
    """Fused transpose + gather: x [N, H, D] (token-major, as a model holds it)
    -> [H, N, D] with row p of every head taken from token perm[p]."""
    x = np.asarray(x)
    return np.ascontiguousarray(np.transpose(x[np.asarray(perm)], (1, 0, 2)))


def restore_heads(o, perm):
    """Inverse of ``reorder_heads``: o [H, N, D] -> y [N, H, D], y[perm[p]] = o[:, p]."""
    o = np.asarray(o)
    y = np.empty((o.shape[1], o.shape[0], o.shape[2]), dtype=o.dtype)
    y[np.asarray(perm)] = np.transpose(o, (1, 0, 2))
    return y


def n_blocks(n: int, B: int) -> int:
    """Number of blocks ceil(n / B) (Section 3.2 "Formulation")."""
    return -(-n // B)


def block_rows(j: int, n: int, B: int) -> slice:
    """Token rows [jB, min(jB + B, n)) of block j."""
    return slice(j * B, min(j * B + B, n))


def block_stats(q, k, v, B: int):
    """Per-block statistics of one head (Section 3.2 "Formulation",
    Eq. (5)-(6); Appendix C "Notation"; Figure 4 "Prepare Phase").

    q, k, v: [n, d] arrays (converted to float64).
    Returns (qbar, kbar, vsum, H, nj):
      qbar[j] = mean of the queries of block j          [nb, d]
      kbar[j] = mean of the keys of block j (centroid)   [nb, d]
      vsum[j] = sum of the values of block j (Vhat_j)    [nb, d]
      H[j]    = sum_n (k_{j,n} - kbar_j)^T v_{j,n}       [nb, d, d]
                (row index: key channel, column index: value channel)
      nj[j]   = number of tokens in block j              [nb]
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, d = q.shape
    nb = n_blocks(n, B)
    qbar = np.empty((nb, d))
    kbar = np.empty((nb, d))
    vsum = np.empty((nb, d))
    H = np.empty((nb, d, d))
    nj = np.empty(nb, dtype=np.int64)
    for j in range(nb):
        r = block_rows(j, n, B)
        nj[j] = r.stop - r.start
        qbar[j] = q[r].mean(axis=0)
        kbar[j] = k[r].mean(axis=0)
        vsum[j] = v[r].sum(axis=0)
        kc = k[r] - kbar[j]
        H[j] = kc.T @ v[r]
    return qbar, kbar, vsum, H, nj


def route_scores(qbar, kbar, scale: float, bias=None, bonus=None):
    """Pooled block scores r_ij = s * qbar_i . kbar_j (Figure 4; Algorithm 1
    step 2 with the plain pooled score), plus a per-key-block term bias_j when
    given (the covariance-aware score of Section 3.3 Eq. 11, see
    ``covariance_bias``) and a per-pair term bonus_ij when given (the
    second-order ranking bonus, see ``second_order_rank_bonus``)."""
    r = scale * (np.asarray(qbar, np.float64) @ np.asarray(kbar, np.float64).T)
    if bias is not None:
        r = r + np.asarray(bias, np.float64)[None, :]
    if bonus is not None:
        r = r + np.asarray(bonus, np.float64)
    return r


def block_heterogeneity(H, Hbar, norm: str = "spectral"):
    """M_j = ||H_j - Hbar|| for every block j (Section 3.3 "Covariance-Aware
    Block Selection" and Theorem 3.1; Appendix D).

    norm="spectral": the largest singular value, the norm written ||.||_2 in
    Section 3.3 and the one Theorem 3.1's bound is stated in. norm="frobenius":
    the Frobenius norm, the variant the Piecewise-Taylor-Attention README uses
    in its router ("hc-free block statistics")."""
    A = np.asarray(H, np.float64) - np.asarray(Hbar, np.float64)[None]
    if norm == "spectral":
        return np.array([np.linalg.svd(a, compute_uv=False)[0] for a in A])
    if norm == "frobenius":
        return np.sqrt((A * A).sum(axis=(1, 2)))
    raise ValueError(norm)


def covariance_bias(M, eps: float):
    """bias_j = log(M_j + eps): the term Eq. 11 adds to the pooled logit of
    key block j. Softmax over j is monotone, and Appendix D's extra -log(Mbar)
    is the same for every j, so ranking by r_ij + bias_j selects the same
    blocks as ranking by Eq. 11 or Eq. 14."""
    return np.log(np.asarray(M, np.float64) + eps)


def route(qbar, kbar, scale: float, topk: int, band: int, bias=None, n_sink: int = 0,
          bonus=None, rows=None):
    """Critical block sets S_i for every query block of one head.

    band(i) = {j : |i - j| <= band}; the first ``n_sink`` key blocks (the
    README's n_sink_blocks, e.g. a text prefix) are forced in as well. The
    remaining blocks are ordered by descending score (``route_scores``, with
    ``bias`` for the covariance-aware variant), lower block index first among
    equal scores, and the first min(topk, #remaining) of them join the forced
    blocks. Returns a list of sorted int64 arrays, one per query block (only
    for the query blocks in ``rows`` when given, in that order).
    """
    nb = np.asarray(kbar).shape[0]
    want = list(range(nb)) if rows is None else list(rows)
    q = np.asarray(qbar, np.float64)[want]
    bon = None if bonus is None else np.asarray(bonus, np.float64)[want]
    r = route_scores(q, kbar, scale, bias, bon)
    sets = []
    idx = np.arange(nb)
    for a, i in enumerate(want):
        forced = (np.abs(idx - i) <= band) | (idx < n_sink)
        in_band = idx[forced]
        cand = idx[~forced]
        # primary key: descending score; secondary key: ascending block index
        order = np.lexsort((cand, -r[a, cand]))
        chosen = cand[order[: min(topk, len(cand))]]
        sets.append(np.sort(np.concatenate([in_band, chosen])).astype(np.int64))
    return sets


def route_gaps(qbar, kbar, scale: float, topk: int, band: int, bias=None, n_sink: int = 0,
               bonus=None, rows=None):
    """Per query block (or per block of ``rows``), the score gap between the
    k-th and (k+1)-th ranked non-forced candidates (inf when the choice is
    forced). Used to recognise near-ties, where several selections are equally
    valid."""
    nb = np.asarray(kbar).shape[0]
    want = list(range(nb)) if rows is None else list(rows)
    bon = None if bonus is None else np.asarray(bonus, np.float64)[want]
    r = route_scores(np.asarray(qbar, np.float64)[want], kbar, scale, bias, bon)
    gaps = np.full(len(want), np.inf)
    idx = np.arange(nb)
    for a, i in enumerate(want):
        cand = r[a, (np.abs(idx - i) > band) & (idx >= n_sink)]
        if 0 < topk < len(cand):
            s = np.sort(cand)[::-1]
            gaps[a] = s[topk - 1] - s[topk]
    return gaps


def second_order_spread(q, k, B: int, scale: float):
    """Second-order correction of the block mass (Piecewise-Taylor-Attention
    README, "Blog post"): for query block i and key block j,
      w_ij = 1/2 * sum_c s^2 mean_{t in i} q_{t,c}^2 * var_{n in j} k_{n,c},
    the per-dimension key variance of block j (over its n_j tokens, 1/n_j)
    weighted by the squared (scaled) queries pooled over query block i, so that
    sum_n exp(q'.k_{j,n}) ~ n_j exp(q'.kbar_j + w_ij). Not gated. [nb, nb]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    n, d = q.shape
    nb = n_blocks(n, B)
    q2 = np.stack([(q[block_rows(i, n, B)] ** 2).mean(axis=0) for i in range(nb)])
    var = np.stack([k[block_rows(j, n, B)].var(axis=0) for j in range(nb)])
    return 0.5 * scale * scale * (q2 @ var.T)


def gate_second_order(w, nj):
    """The README's gate: where w_ij exceeds ln(n_j) (the largest mass gain the
    expansion may claim for a block of n_j tokens) the term is set to 0 and the
    block falls back to the zeroth-order mass; elsewhere w_ij is kept."""
    w = np.asarray(w, dtype=np.float64)
    lim = np.log(np.asarray(nj, dtype=np.float64))[None, :]
    return np.where(w > lim, 0.0, w)


def second_order_rank_bonus(w, nj):
    """The README's ranking use of the spread ("Router polish"): the bounded
    bonus min(w_ij, ln n_j) added to the pooled route score, so a block whose
    expansion saturates still ranks with the largest admissible gain, while the
    forward uses the gated spread (``gate_second_order``)."""
    w = np.asarray(w, dtype=np.float64)
    return np.minimum(w, np.log(np.asarray(nj, dtype=np.float64))[None, :])


def forward(q, k, v, B: int, scale: float, sets, stats=None, qblocks=None,
            first_order: bool = True, spread=None):
    """Piecewise forward of one head (Section 3.2, Eq. (3)-(6)).

    For each query t of query block i, with q' = s * q_t:
      D_t = sum_{j in S_i} sum_n exp(q'.k_{j,n} - m)
            + sum_{j in U_i} n_j exp(q'.kbar_j - m)
      N_t = sum_{j in S_i} sum_n exp(q'.k_{j,n} - m) v_{j,n}
            + sum_{j in U_i} exp(q'.kbar_j - m) (Vhat_j + q' H_j)
      o_t = N_t / D_t
    The first-order term in the denominator vanishes because the centred keys
    of a block sum to zero (remark under Eq. (6)), so the block mass is
    n_j exp(q'.kbar_j).

    sets: list of critical block index arrays (from ``route`` or supplied).
    stats: optional precomputed ``block_stats`` result.
    qblocks: iterable of query block indices to evaluate (default: all).
    first_order: False drops the Eq. (6) term (zeroth-order variant); used by
      the convergence-order check only.
    spread: optional [nb, nb] matrix w_ij (``gate_second_order`` of
      ``second_order_spread``) added to the logit of every approximated block,
      the second-order "virtual token" of the Piecewise-Taylor-Attention
      README: mass n_j exp(a + w), numerator exp(a + w) (Vhat_j + q' H_j).
    Returns {i: [rows_i, d] float64 output} when qblocks is given, else the
    full [n, d] array.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, d = q.shape
    nb = n_blocks(n, B)
    if stats is None:
        stats = block_stats(q, k, v, B)
    _, kbar, vsum, H, nj = stats
    want = range(nb) if qblocks is None else qblocks
    out = {}
    for i in want:
        rows = block_rows(i, n, B)
        qp = scale * q[rows]  # q' = s q
        S = np.asarray(sets[i], dtype=np.int64)
        sel = np.zeros(nb, dtype=bool)
        sel[S] = True
        U = np.nonzero(~sel)[0]
        # exact logits over the selected blocks
        ks = np.concatenate([k[block_rows(j, n, B)] for j in S]) if len(S) else np.zeros((0, d))
        vs = np.concatenate([v[block_rows(j, n, B)] for j in S]) if len(S) else np.zeros((0, d))
        e = qp @ ks.T  # [m, sum n_j]
        a = qp @ kbar[U].T  # centroid logits [m, |U|]
        if spread is not None:
            a = a + np.asarray(spread, dtype=np.float64)[i, U][None, :]
        m = np.full(qp.shape[0], -np.inf)
        if e.shape[1]:
            m = np.maximum(m, e.max(axis=1))
        if a.shape[1]:
            m = np.maximum(m, a.max(axis=1))
        pe = np.exp(e - m[:, None])
        alpha = np.exp(a - m[:, None])
        den = pe.sum(axis=1) + alpha @ nj[U].astype(np.float64)
        num = pe @ vs + alpha @ vsum[U]
        if first_order and len(U):
            # sum_j alpha_tj (q'_t H_j): the [m, |U| d] x [|U| d, d] product of
            # the row-wise outer products alpha_t (x) q'_t with the stacked H_j.
            w = (alpha[:, :, None] * qp[:, None, :]).reshape(qp.shape[0], -1)
            num = num + w @ H[U].reshape(-1, d)
        out[i] = num / den[:, None]
    if qblocks is not None:
        return out
    return np.concatenate([out[i] for i in range(nb)], axis=0)


def forward_head(q, k, v, B: int, scale: float, topk: int, band: int,
                 qblocks=None):
    """Stats, route and forward of one head in one call. Returns
    (output, sets, stats)."""
    stats = block_stats(q, k, v, B)
    sets = route(stats[0], stats[1], scale, topk, band)
    o = forward(q, k, v, B, scale, sets, stats=stats, qblocks=qblocks)
    return o, sets, stats


def global_first_order(H):
    """Hbar = (1/n_b) sum_j H_j: the query-independent global first-order
    statistic of the hybrid approximation (Section 3.3, Eq. 10; Appendix C
    "Notation")."""
    return np.asarray(H, dtype=np.float64).mean(axis=0)


def forward_hybrid(q, k, v, B: int, scale: float, sets, stats=None, qblocks=None):
    """Hybrid-order forward of one head (Section 3.3, Eq. 9-10; Algorithm 1).

    For each query t of query block i, with q' = s * q_t and
    alpha_tj = exp(q'.kbar_j - m):
      D_t = sum_{j in S_i} sum_n exp(q'.k_{j,n} - m) + sum_{j in U_i} n_j alpha_tj
      N_t = sum_{j in S_i} sum_n exp(q'.k_{j,n} - m) v_{j,n}
            + sum_{j in U_i} alpha_tj Vhat_j + (sum_{j in U_i} alpha_tj) q' Hbar
      o_t = N_t / D_t
    Arguments and return value as for ``forward``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, d = q.shape
    nb = n_blocks(n, B)
    if stats is None:
        stats = block_stats(q, k, v, B)
    _, kbar, vsum, H, nj = stats
    Hbar = global_first_order(H)
    want = range(nb) if qblocks is None else qblocks
    out = {}
    for i in want:
        rows = block_rows(i, n, B)
        qp = scale * q[rows]
        S = np.asarray(sets[i], dtype=np.int64)
        sel = np.zeros(nb, dtype=bool)
        sel[S] = True
        U = np.nonzero(~sel)[0]
        ks = np.concatenate([k[block_rows(j, n, B)] for j in S]) if len(S) else np.zeros((0, d))
        vs = np.concatenate([v[block_rows(j, n, B)] for j in S]) if len(S) else np.zeros((0, d))
        e = qp @ ks.T
        a = qp @ kbar[U].T
        m = np.full(qp.shape[0], -np.inf)
        if e.shape[1]:
            m = np.maximum(m, e.max(axis=1))
        if a.shape[1]:
            m = np.maximum(m, a.max(axis=1))
        pe = np.exp(e - m[:, None])
        alpha = np.exp(a - m[:, None])
        den = pe.sum(axis=1) + alpha @ nj[U].astype(np.float64)
        num = pe @ vs + alpha @ vsum[U] + alpha.sum(axis=1)[:, None] * (qp @ Hbar)
        out[i] = num / den[:, None]
    if qblocks is not None:
        return out
    return np.concatenate([out[i] for i in range(nb)], axis=0)
