"""bench.py's multi-rank path on CPU: two gloo ranks (one process each),
as torchrun launches them on a node.  Requests are independent, so each
rank verifies its own batch; the job's throughput counts every rank's
requests over the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys

    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [0.50, 0.80][rank]             # rank 1 is the slower one
        mx = bench.reduce_max(elapsed, dist, "cpu")
        out[rank] = (mx, bench.job_throughput(64, world, 10, mx))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        mx, value = res[r]
        assert mx == pytest.approx(0.80)
        assert value == pytest.approx(2 * 64 * 10 / 0.80)


def test_single_process_needs_no_group():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max(0.25, None, "cpu") == 0.25
    assert bench.job_throughput(64, 1, 4, 0.5) == pytest.approx(512.0)


def test_ranks_get_distinct_workload_seeds():
    """Each rank builds its own batch (weak scaling): the seeds differ."""
    from speculative_decoding_verification_23_gb300 import workload as W

    a = W.make_batch(B=2, V=64, K=2, seed=3 * 10 ** 6 + 0, hist_len=4)
    b = W.make_batch(B=2, V=64, K=2, seed=3 * 10 ** 6 + 1, hist_len=4)
    assert not (a.target == b.target).all()
