"""The benchmark's multi-rank path on CPU: two gloo ranks, as `torchrun --nproc-per-node 2 bench.py` runs them.

The operator shards into independent replicas (no exchange step), so the only cross-rank logic is host
side: the barrier around the timed region, the maximum of the per-rank step times, and rank 0 alone
printing (and, for the oracle arm, doing) the work.
"""

import argparse
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist

    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    bench.dist_init(w)
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.0 + rank, w)           # rank 1 is the slower replica
    args = argparse.Namespace(workload="prefill_8k", warmup=3, steps=1)
    ref_line = bench.run_reference(args, rank, w) if rank != 0 else "rank0"
    out.put((rank, slowest, ref_line))
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(world))
    assert [g[1] for g in got] == [2.0, 2.0]
    assert got[1][2] is None            # only rank 0 runs the oracle arm and prints its line


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
