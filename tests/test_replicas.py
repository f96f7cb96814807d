"""The benchmark's replica bookkeeping on two gloo ranks on the CPU: the drafter's round
does not shard (sequences are independent), so N GPUs run N replicas and the only
cross-rank work is timing -- a barrier, the slowest rank's time and the sum of tokens."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        tokens = 100.0 * (rank + 1)            # rank r drafted 100 (r + 1) tokens
        elapsed = 10.0 + 30.0 * rank           # in 10 + 30 r ms
        value, t = bench.replica_throughput(world, tokens, elapsed)
        out[rank] = (value, t, bench.max_over_ranks(world, float(rank)),
                     bench.sum_over_ranks(world, 1.0))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_tokens_over_the_slowest_time():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        value, t, mx, sm = out[r]
        assert t == 40.0                       # the slowest rank
        assert abs(value - 300.0 / 0.040) < 1e-6   # 300 tokens in 40 ms
        assert mx == 1.0 and sm == 2.0


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_throughput(1, 300.0, 40.0) == (300.0 / 0.040, 40.0)
    assert bench.max_over_ranks(1, 3.5) == 3.5 and bench.sum_over_ranks(1, 2.0) == 2.0
