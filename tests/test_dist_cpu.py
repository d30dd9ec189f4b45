"""The N>1 host logic of bench.py on CPU: two gloo ranks agree on the max
step time, and the barrier helper works without a GPU."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench._dist_env() == (world, rank, rank)
        bench.barrier()
        out[rank] = bench.max_over_ranks(1.5 + 3.0 * rank)
        bench.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 4.5, 1: 4.5}


def test_max_without_process_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(2.25) == 2.25
