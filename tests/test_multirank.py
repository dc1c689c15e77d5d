"""The benchmark's multi-rank host logic on CPU: two gloo ranks (no GPU).

Each rank of `bench.py --gpus N` runs an independent replica of the workload
(the path has no exchange step), the slowest rank's time is the job's time, and
the whole-job value counts every rank's bytes.  The reference arm runs on rank 0
only.
"""

import os
import socket
import sys
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank step times: the job's time is the largest
        ms = bench.max_over_ranks(1.0 + 2.5 * rank, world, torch.device("cpu"))
        total = bench.whole_job_gbps(world, 1_000_000, ms)
        dist.barrier()
        # the reference arm does nothing on ranks other than 0
        args = types.SimpleNamespace(config=1, steps=1, warmup=3)
        if rank != 0:
            assert bench.run_reference(args, world, rank) is None
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ms!r} {total!r}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_bytes(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True, start_method="spawn")
    vals = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    for ms, total in vals:
        assert float(ms) == 3.5                                  # max(1.0, 3.5)
        assert float(total) == pytest.approx(2 * 1e6 / 3.5e-3 / 1e9)


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, 1, None) == 4.25
    assert bench.whole_job_gbps(1, 2_000_000, 2.0) == pytest.approx(1.0)
