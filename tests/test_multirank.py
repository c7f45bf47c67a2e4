"""The N > 1 host path of bench.py on the CPU with two gloo ranks: whole-job
throughput uses the slowest rank's time, the max reaches every rank, and the
reference arm runs on rank 0 only."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, _ = bench.dist_setup()
    assert (r, w) == (rank, world)
    value = bench.aggregate_throughput(1000, 1.0 + rank, world)   # rank 1 takes 2 s
    slowest = bench.max_over_ranks(3.0 * rank, world)
    bench.barrier(world)
    import argparse
    ref = bench.bench_reference(argparse.Namespace(workload=bench.HEADLINE, steps=1, warmup=0), rank, world) \
        if rank != 0 else "rank0"
    q.put((rank, value, slowest, ref))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, slowest, ref in out:
        assert value == 1000 * 2 / 2.0      # units of both ranks / slowest rank's seconds
        assert slowest == 3.0
    assert out[1][3] is None                # the reference arm does no work off rank 0
