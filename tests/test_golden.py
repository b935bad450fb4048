"""Hand-worked fixtures under tests/golden/ (each file cites the equations its
values were derived from) checked against the fp64 oracle."""

import json
import os

import numpy as np

from oracle import block_stats, forward, route, route_gaps

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_piecewise_d1_hand_examples():
    data = load("piecewise_d1.json")
    for case in data["cases"]:
        col = lambda key: np.array(case[key], dtype=np.float64)[:, None]
        q, k, v = col("q"), col("k"), col("v")
        B, s = case["block"], case["scale"]
        st = block_stats(q, k, v, B)
        o = forward(q, k, v, B, s, [np.array(x, dtype=np.int64) for x in case["sets"]], stats=st)
        np.testing.assert_allclose(o[:, 0], case["expected"], rtol=1e-14, atol=1e-14,
                                   err_msg=case["name"])


def test_route_ties_hand_example():
    data = load("route_ties.json")
    qbar = np.array(data["qbar"], dtype=np.float64)
    kbar = np.array(data["kbar"], dtype=np.float64)
    sets = route(qbar, kbar, data["scale"], data["topk"], data["band"])
    assert [list(map(int, s)) for s in sets] == data["expected"]


def test_route_gaps_hand_example():
    """Selection margins worked by hand from integer block means (exact scores):
    a plain top-k, a band, a sink block with a per-key-block bias, ties at the
    boundary (margin 0) and rows with nothing left to choose (margin inf)."""
    data = load("route_gaps.json")
    qbar = np.array(data["qbar"], dtype=np.float64)
    kbar = np.array(data["kbar"], dtype=np.float64)
    np.testing.assert_array_equal(qbar @ kbar.T, np.array(data["unscaled_scores"], np.float64))
    for case in data["cases"]:
        bias = None if case["bias"] is None else np.array(case["bias"], dtype=np.float64)
        got = route_gaps(qbar, kbar, case["scale"], case["topk"], case["band"], bias=bias,
                         n_sink=case["n_sink"])
        want = np.array([np.inf if x == "inf" else x for x in case["expected"]], np.float64)
        np.testing.assert_array_equal(got, want, err_msg=case["name"])
        # the same margins for a subset of rows, in another order
        rows = [5, 0, 3]
        sub = route_gaps(qbar, kbar, case["scale"], case["topk"], case["band"], bias=bias,
                         n_sink=case["n_sink"], rows=rows)
        np.testing.assert_array_equal(sub, want[rows], err_msg=case["name"])
