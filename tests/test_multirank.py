"""The benchmark's multi-rank host logic, run as two gloo ranks on the CPU.

Under torchrun every rank times its own copy of the workload on its own GPU
(independent problems, no collective on the data path); the ranks meet only
at a barrier around the timed region and in one max-reduction of the elapsed
time.  These tests run that plumbing with world size 2 on the gloo backend:
no GPU is involved.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        env = bench.dist_env()
        # each rank reports its own elapsed time; the slowest one is used
        slowest = bench.max_over_ranks(10.0 + 3.0 * rank, world, torch.device("cpu"))
        bench.barrier(world)
        # only rank 0 runs the reference arm; the others return at once
        args = type("A", (), {"gpus": world, "steps": 1, "warmup": 3})()
        ref_rc = bench.run_reference(args) if rank != 0 else 0
        out.put((rank, env, slowest, ref_rc))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True,
                       start_method="spawn")
    got = sorted(out.get() for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    for rank, env, slowest, ref_rc in got:
        assert env == (2, rank, rank)
        assert slowest == 13.0          # max over ranks, seen by every rank
        assert ref_rc == 0


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(4.5, 1, torch.device("cpu")) == 4.5
    bench.barrier(1)  # no-op without torch.distributed


@pytest.mark.parametrize("world", [1, 2, 4, 8])
def test_job_throughput_is_weak_scaling_over_ranks(world):
    f_fwd, f_bwd = bench.flops(1, 32, 8192, 128, True)
    step = f_fwd + f_bwd
    # every rank processes one full workload per step in the slowest rank's time
    assert bench.job_tflops(world, step, 1.5) == pytest.approx(world * step / 1.5e-3 / 1e12)
    assert bench.job_tflops(world, step, 1.5) == pytest.approx(world * bench.job_tflops(1, step, 1.5))


def test_headline_flop_convention():
    # forward 4*B*H*N^2*d halved for causal, backward 2.5x the forward
    f_fwd, f_bwd = bench.flops(1, 32, 8192, 128, True)
    assert f_fwd == 4 * 32 * 8192 ** 2 * 128 / 2
    assert f_bwd == 2.5 * f_fwd
