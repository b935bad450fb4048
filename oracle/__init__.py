"""fp64 CPU reference for piecewise sparse attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product package.
"""

from .pisa_oracle import (  # noqa: F401
    block_heterogeneity,
    block_rows,
    block_stats,
    covariance_bias,
    forward,
    forward_head,
    forward_hybrid,
    gate_second_order,
    global_first_order,
    morton_permutation,
    n_blocks,
    reorder_heads,
    restore_heads,
    route,
    route_gaps,
    route_scores,
    second_order_rank_bonus,
    second_order_spread,
)
