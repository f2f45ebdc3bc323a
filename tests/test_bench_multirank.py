"""The multi-rank path of bench.py on CPU: two gloo ranks.

bench.py runs one independent replica of the workload per GPU (the path has
no exchange step) and reports the slowest rank's time and the whole-job
throughput. These tests check that arithmetic with real torch.distributed
ranks over gloo on 127.0.0.1, no GPU involved.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        slowest = bench.max_over_ranks(times[rank], world)
        value = bench.whole_job_tflops(world, 1e12, slowest)
        with open(f"{out_path}.{rank}", "w") as f:
            f.write(f"{slowest} {value}\n")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(2.0, 5.0), (7.5, 1.25)])
def test_two_rank_max_and_whole_job_value(tmp_path, times):
    world = 2
    out = str(tmp_path / "r")
    mp.start_processes(_rank_main, args=(world, _free_port(), times, out), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        slowest, value = map(float, open(f"{out}.{r}").read().split())
        assert slowest == max(times)
        # 1e12 FLOPs per rank per step, both ranks: 2e12 / (max ms * 1e-3) / 1e12
        assert value == pytest.approx(world * 1e12 / (max(times) * 1e-3) / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.whole_job_tflops(1, 2e12, 4.0) == pytest.approx(500.0)
