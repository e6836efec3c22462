"""The N > 1 host path of bench.py on CPU: two gloo ranks (replicas, no
data-path collective). The job's time is the slowest rank's, the job's
throughput counts every rank's tokens, and only rank 0 prints."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        got = bench.max_over_ranks(10.0 + 5.0 * rank, dist, torch.device("cpu"))
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn")
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, torch.device("cpu")) == 3.5
    # two replicas of 8192 tokens, 10 steps in 20 ms: 2 * 8192 * 10 / 0.02
    assert bench.tokens_per_s(2, 8192, 10, 20.0) == pytest.approx(8192000.0)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_roofline_bound_follows_the_ridge():
    """The Switch-shaped FFN (111 FLOP per byte) is HBM-bound; the Mixtral-
    and DeepSeek-shaped ones are tensor-bound and, at milliseconds per call,
    measured against the sustained bf16 rate."""
    import bench
    pk = {"hbm_gbs": 6490.5, "bf16_tflops": 1744.3, "bf16_tflops_sustained": 1392.1}
    sw = bench.roofline_record(137e9, 1.235e9, 0.203, pk, "measured", 605e6)
    assert sw["bound"] == "hbm" and sw["unit"] == "GB/s" and sw["traffic"] == 605e6
    assert abs(sw["achieved"] - 1.235e9 / 0.203e-3 / 1e9) < 1e-6
    assert abs(sw["frac"] - sw["achieved"] / 6490.5) < 1e-12
    mx = bench.roofline_record(11.54e12, 3.6e9, 9.4, pk, "measured", None)
    assert mx["bound"] == "tensor" and mx["unit"] == "TFLOP/s"
    assert mx["peak"] == 1392.1 and mx["peak_kind"] == "measured sustained"
    assert abs(mx["achieved"] - 11.54e12 / 9.4e-3 / 1e12) < 1e-9
    short = bench.roofline_record(11.54e12 / 20, 3.6e9 / 20, 0.47, pk, "fallback", None)
    assert short["peak"] == 1744.3 and short["peak_kind"] == "fallback burst"
    # DeepSeek-shaped: 256 FLOP per byte, below the burst ridge (269) but above
    # the sustained one (214); at milliseconds per call the FLOPs bind
    ds = bench.roofline_record(6.49e12, 25.3e9, 7.37, pk, "measured", None)
    assert ds["bound"] == "tensor" and ds["peak"] == 1392.1
