"""The multi-GPU bench path runs independent replicas; its host logic (process group, max-over-ranks
time, whole-job rate) checked with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as tmp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r timed (100 + 50 r) ms for 64 steps: the job takes the slowest rank's time
    value, total_ms = bench.whole_job_rate(100.0 + 50.0 * rank, 64, world, dist)
    dist.barrier()
    with open(f"{out_path}.{rank}", "w") as f:
        f.write(f"{value} {total_ms}\n")
    dist.destroy_process_group()


def test_whole_job_rate_two_ranks(tmp_path):
    world, port = 2, _free_port()
    out = str(tmp_path / "rate")
    tmp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        value, total_ms = map(float, open(f"{out}.{r}").read().split())
        assert total_ms == pytest.approx(150.0)
        assert value == pytest.approx(world * 64 / 0.150)


def test_whole_job_rate_single():
    import bench
    value, total_ms = bench.whole_job_rate(200.0, 100, 1, None)
    assert total_ms == 200.0 and value == pytest.approx(500.0)
