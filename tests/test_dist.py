"""Multi-rank host logic of bench.py on CPU with the gloo backend (2 ranks):
per-rank replicas draw different inputs and the reported time is the maximum
over ranks. No GPU and no data-path collective are involved."""

import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from piecewise_sparse_attention_gb300.workloads import WORKLOADS, make_head

        vals = bench.max_over_ranks([1.0 + rank, 5.0 - rank])
        q, _, _ = make_head(WORKLOADS["tiny"], 0, seed_offset=bench.rank_seed_offset(rank))
        out[rank] = (vals, float(q[:4, :4].sum()))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction_and_replicas():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    (v0, s0), (v1, s1) = out[0], out[1]
    assert v0 == v1 == [2.0, 5.0]
    assert s0 != s1  # each rank draws its own replica


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert np.isclose(bench.rank_seed_offset(0), 0)
