"""bench.py's multi-rank plumbing on CPU: two gloo ranks, max-over-ranks timing and the
whole-job aggregate (units of every rank over the slowest rank's time)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [40.0, 55.0][rank]                       # rank 1 is the slow one
        m = bench.max_over_ranks(ms, world)
        bench.barrier(world)
        out[rank] = (m, bench.aggregate_rate(32 * 100, world, m))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_units():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as man:
        out = man.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs)
        res = dict(out)
    for r in range(world):
        m, v = res[r]
        assert m == 55.0
        assert v == pytest.approx(32 * 100 * 2 / 0.055)


def test_single_rank_is_its_own_maximum():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_rate(10, 1, 1000.0) == pytest.approx(10.0)



def test_launch_counts_per_step():
    """The gpu_launches claim: append, Full select (clear, scan, [collect,] finalize), three per
    Reindex (clear, score, select), one attention per layer, and with draft rows three more
    per indexer layer for the rows' own selection."""
    sys.path.insert(0, ROOT)
    import bench
    from synth.workloads import config, verify_workload
    assert bench.kernels_per_step(config(1)) == 1 + 3 + 4                  # 8192 blocks: no collect
    assert bench.kernels_per_step(config(2)) == 1 + 4 + 3 * 4 + 20         # 131072 blocks: collect
    v = verify_workload()
    assert v.drafts == 5 and v.ring >= v.window + v.drafts - 1
    assert bench.kernels_per_step(v) == 1 + 3 + 3 * 5 + 20
