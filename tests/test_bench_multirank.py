"""The benchmark's replica path on two CPU ranks (gloo): every rank measures its
own replica, the job time is the slowest rank's, and the whole-job value counts
every rank's bytes. No GPU and no data-path collective are involved: the op
does not shard, and the only exchange is this timing maximum."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_path: str):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")  # rank 1 is slower
        value = bench.job_gbps(4_000_000, world, slowest)
        with open(f"{out_path}.{rank}", "w") as f:
            f.write(f"{slowest} {value}")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step(tmp_path):
    world = 2
    out = str(tmp_path / "res")
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        slowest, value = map(float, open(f"{out}.{r}").read().split())
        assert slowest == 15.0
        # 2 ranks x 4 MB over 15 ms
        assert value == pytest.approx(2 * 4e6 / 15e-3 / 1e9)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.job_gbps(1_000_000_000, 1, 1000.0) == pytest.approx(1.0)


def test_launch_count_follows_the_plan():
    import bench
    import decode_attention_04_gb300 as fd
    p = fd.fd_plan_sms(1, 16, 8, 256, 1024, 1024, 0, 152, 2, 8)
    assert bench.kernels_per_call(p) == 2          # split + merge
    fd.fd_plan_override(p, 16, 0, 16, -1)
    assert bench.kernels_per_call(p) == 1          # one cluster spans the band
    fd.fd_plan_override(p, 32, 0, 1, 1)
    assert bench.kernels_per_call(p) == 1          # fused merge
