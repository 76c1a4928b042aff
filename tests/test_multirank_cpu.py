"""The bench's multi-process path on CPU: two ranks over gloo (127.0.0.1).

The layer shards as independent replicas (one GPU per rank, no collective on
the data path); the only cross-rank steps are the barrier around the timed
region and the max over ranks of the step time. This checks those helpers
with real processes and a real process group, and that the reference arm
runs on rank 0 only.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench.max_over_ranks(dist, times[rank], "cpu")
        value = bench.job_throughput(ws, 4096, slowest)

        class Args:
            workload, tokens, fwd_only, cpu_sample_tokens, warmup, steps = (
                "tiny_fp32", 0, False, 3, 0, 1)
        ref = bench.run_reference(Args, ws, rank)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{slowest} {value} {ref is not None}\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_rank0_reports(tmp_path):
    times = [3.25, 7.5]
    mp.start_processes(_worker, args=(2, _free_port(), times, str(tmp_path)), nprocs=2,
                       join=True, start_method="spawn")
    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(2)]
    for slowest, value, _ in rows:
        assert float(slowest) == 7.5
        # both ranks' tokens over the slowest rank's step
        assert float(value) == round(2 * 4096 / 7.5e-3, 1)
    assert rows[0][2] == "True" and rows[1][2] == "False"


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(None, 2.5, "cpu") == 2.5
    assert bench.job_throughput(1, 1000, 2.0) == 500000.0
