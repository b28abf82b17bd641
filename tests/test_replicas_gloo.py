"""The multi-GPU benchmark path on CPU: replicas only (the draft head does not
shard on one box), so the only exchange is the max-over-ranks timing. Two gloo
ranks check that every rank sees the slowest rank's time and that the
whole-job value counts the steps of all replicas."""
import os
import socket

import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 20.0][rank]
        got = bench.max_over_ranks(local_ms, torch.device("cpu"))
        value = bench.whole_job_us_per_step(got, 1000, world)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{got} {value}")
    finally:
        tdist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_replicas_agree_on_the_slowest_time(tmp_path):
    mp.start_processes(_rank, args=(2, _free_port(), str(tmp_path)), nprocs=2, start_method="spawn")
    for r in range(2):
        got, value = map(float, open(tmp_path / f"rank{r}.txt").read().split())
        assert got == 20.0
        assert value == pytest.approx(20.0e3 / 2000)   # 2 x 1000 steps in 20 ms


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.25, torch.device("cpu")) == 3.25
    assert bench.whole_job_us_per_step(20.5, 1000, 1) == pytest.approx(20.5)
