"""Replicas: `bench.py --gpus N` runs one independent replica per rank (the
path shards by 128-row tiles but needs no exchange), takes the slowest rank's
time and reports whole-job throughput.  The cross-rank pieces are checked here
on CPU with two gloo ranks."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, result_dir: str):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) * 1.5 ms: every rank must see the slowest
        got = bench.max_over_ranks((rank + 1) * 1.5, "cpu")
        with open(os.path.join(result_dir, f"rank{rank}"), "w") as f:
            f.write(repr(got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        assert float((tmp_path / f"rank{r}").read_text()) == pytest.approx(3.0)


def test_max_over_ranks_without_a_group_is_the_value():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, "cpu") == 2.5


def test_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    # 340.8 M weights per replica in 0.1 ms: 6816 GB/s for one, twice for two
    one = bench.job_weight_gbs(340_800_000, 1, 0.1)
    assert one == pytest.approx(6816.0)
    assert bench.job_weight_gbs(340_800_000, 2, 0.1) == pytest.approx(2 * one)
