"""CPU checks of the near-tie rule the GPU route tests share (route_check.py):
on the hand-worked margins of tests/golden/route_gaps.json, a different but
equally valid selection at a tie is accepted, and every kind of invalid
selection is rejected."""

import json
import os

import numpy as np
import pytest

import oracle
from route_check import check_route_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "route_gaps.json")


@pytest.fixture(scope="module")
def means():
    with open(GOLDEN) as f:
        data = json.load(f)
    return np.array(data["qbar"], np.float64), np.array(data["kbar"], np.float64)


def sets_of(qbar, kbar, *a, **kw):
    return [list(map(int, x)) for x in oracle.route(qbar, kbar, *a, **kw)]


def test_oracle_route_passes(means):
    qbar, kbar = means
    got = sets_of(qbar, kbar, 0.5, 2, 0)
    used, ties = check_route_rows(got, qbar, kbar, 0.5, 2, 0)
    assert ties == 0 and [list(u) for u in used] == got


def test_other_choice_at_a_tie_passes(means):
    qbar, kbar = means
    got = sets_of(qbar, kbar, 0.5, 2, 0)
    assert got[4] == [0, 1, 4]          # every score of row 4 is 0: any two free blocks
    got[4] = [0, 4, 5]
    used, ties = check_route_rows(got, qbar, kbar, 0.5, 2, 0)
    assert ties == 1 and list(used[4]) == [0, 4, 5]


@pytest.mark.parametrize("row,bad", [
    (0, [0, 1, 4]),        # row 0 has margin 0.5: only {1, 2} is valid
    (4, [0, 1, 2]),        # the band block 4 dropped
    (4, [0, 1, 3, 4]),     # one block too many
    (4, [1, 0, 4]),        # not ascending
    (4, [0, 0, 4]),        # a repeat
])
def test_invalid_choice_fails(means, row, bad):
    qbar, kbar = means
    got = sets_of(qbar, kbar, 0.5, 2, 0)
    got[row] = bad
    with pytest.raises(AssertionError):
        check_route_rows(got, qbar, kbar, 0.5, 2, 0)


def test_tie_with_sink_and_bias(means):
    """Row 1 of the sink + bias case ties j = 2 and j = 3 at the boundary; a
    pick below the tie value (j = 4) is rejected, the other tied block passes,
    and dropping the sink block 0 is rejected."""
    qbar, kbar = means
    bias = np.array([0, 0.25, -1, 2, 0, 0.5])
    kw = dict(bias=bias, n_sink=1)
    got = sets_of(qbar, kbar, 1.0, 2, 0, **kw)
    assert got[1] == [0, 1, 2, 5]
    alt = [row[:] for row in got]
    alt[1] = [0, 1, 3, 5]
    assert check_route_rows(alt, qbar, kbar, 1.0, 2, 0, **kw)[1] == 1
    for bad in ([0, 1, 4, 5], [1, 2, 3, 5]):
        alt[1] = bad
        with pytest.raises(AssertionError):
            check_route_rows(alt, qbar, kbar, 1.0, 2, 0, **kw)


def test_row_subset(means):
    qbar, kbar = means
    rows = [5, 2]
    got = [list(map(int, x)) for x in oracle.route(qbar, kbar, 1.0, 1, 1, rows=rows)]
    used, ties = check_route_rows(got, qbar, kbar, 1.0, 1, 1, rows=rows)
    assert ties == 0 and len(used) == 2
