"""The bench's multi-rank path on CPU: two gloo ranks stand in for two GPUs running
independent replicas (weak scaling, no collective on the data path).  Each rank times
its own work; the reported time is the slowest rank's and the value counts every rank's
units.  The reference arm runs on rank 0 only.  No GPU."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [12.5, 20.0][rank]                        # rank 1 is the slower replica
        worst = bench.max_over_ranks(my_ms, torch.device("cpu"))
        value = bench.whole_job_rate(1.0e9, world, worst)
        # the reference arm: rank 0 alone runs and prints; the others return at once
        class Args:
            workload, ref_seqs, warmup, steps = "gqa70b", 1, 0, 1
        buf = io.StringIO()
        with redirect_stdout(buf):
            if rank != 0:
                bench.bench_reference(Args())
        q.put((rank, worst, value, bench.dist_env(), buf.getvalue()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_every_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, value, env, printed in results:
        assert worst == 20.0                              # both ranks agree on the max
        assert value == pytest.approx(1.0e9 * 2 / 0.020)  # both replicas' units
        assert env == (2, rank, rank)
        assert printed == ""                              # rank 1's reference arm did nothing
