"""The N>1 host logic of bench.py on CPU: two gloo ranks agree on the max
step time, the barrier helper works without a GPU, and `bench.py --gpus 2`
starts its own two ranks (here in its CPU-only dry-run mode, on gloo), both
of which report to rank 0."""
import json
import os
import socket
import subprocess
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
    # the manager process is spawned too: this test process may already run
    # threads (the OpenMP oracle), and a fork from a threaded process can hang
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 4.5, 1: 4.5}


def test_max_without_process_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(2.25) == 2.25


def _run_bench(*args, env=None):
    e = {k: v for k, v in os.environ.items()
         if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=300, env=e, cwd=ROOT)


def test_bench_launches_its_own_ranks():
    """--gpus 2 without torchrun: bench.py starts ranks 0 and 1 itself; only
    rank 0 prints, and the line counts both ranks."""
    p = _run_bench("--gpus", "2", "--dry-run", "--steps", "3", "--warmup", "3")
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(x) for x in p.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = lines[0]
    assert line["dry_run"] is True and line["value"] is None
    assert line["n_gpus"] == 2
    assert line["ranks_reported"] == [0, 1] and line["local_ranks"] == [0, 1]


def test_bench_single_rank_dry_run():
    p = _run_bench("--dry-run", "--steps", "2")
    assert p.returncode == 0, p.stderr[-2000:]
    line = json.loads(p.stdout.strip().splitlines()[-1])
    assert line["n_gpus"] == 1 and line["ranks_reported"] == [0]


def test_bench_launcher_reports_a_failing_rank():
    """A rank that fails makes the launcher fail (here: an unknown argument
    in every rank)."""
    p = _run_bench("--gpus", "2", "--dry-run", "--steps", "nope")
    assert p.returncode != 0
