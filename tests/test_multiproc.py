"""The N > 1 path of bench.py on the CPU: two gloo ranks.

The op runs as independent replicas (no data-path collective); the only
collectives are the barrier around the timed region and the max over ranks
of the step time.  Both are exercised here, and the reference arm's rule
that only rank 0 does work.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    dist = bench.dist_init(w, use_cuda=False)
    bench.barrier(dist)
    step_ms = 1.0 + 1.5 * rank           # rank 1 is the slow one
    got = bench.max_over_ranks(dist, step_ms, "cpu")
    bench.barrier(dist)
    dist.destroy_process_group()
    out[rank] = got


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_barrier(world):
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_reference_arm_does_nothing_on_other_ranks():
    sys.path.insert(0, ROOT)
    import bench

    class A:
        workload = "toy"
        steps = 1
        warmup = 3
    assert bench.run_reference(A(), rank=1, world=2) == 0
