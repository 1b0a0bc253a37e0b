"""The benchmark's multi-rank path on CPU: world size 2 over gloo (no GPU).

Each rank runs an independent replica of the verify step (requests are
independent; nothing is exchanged on the data path), so the whole-job value
is the sum of the ranks' accepted tokens over the slowest rank's time. Here
each rank reports a made-up token count and time and the reduction is checked.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        tokens = [300.0, 500.0][rank]
        t_ms = [100.0, 250.0][rank]
        value, t_max = bench.aggregate(tokens, t_ms, world)
        bench.barrier(world)
        out[rank] = (value, t_max)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_sum_tokens_over_slowest_time():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        value, t_max = out[r]
        assert t_max == 250.0
        assert abs(value - 800.0 / 0.25) < 1e-9


def test_single_rank_is_identity():
    import bench
    value, t_max = bench.aggregate(123.0, 10.0, 1)
    assert t_max == 10.0 and abs(value - 12300.0) < 1e-9
