"""The multi-process (torchrun) path of bench.py on CPU with gloo, world size 2.

The GEMM does not shard here: each rank runs an independent replica, so the
only cross-rank logic is the barrier around the timed region, the max over
ranks of its length, and the whole-job throughput (all ranks' flops over the
slowest rank's time).  No GPU.
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


def _worker(rank, world, port, local_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        m = bench.slowest_rank_ms(local_ms[rank], dist, "cpu")
        out[rank] = m
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_replica_throughput_gloo_world2():
    world = 2
    local_ms = [120.0, 150.5]
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), local_ms, out), nprocs=world, join=True)
    assert out[0] == out[1] == 150.5
    flops = 2.0 * 8192 ** 3
    v = bench.replicas_tflops(world, flops, 10, out[0])
    assert v == pytest.approx(world * flops * 10 / 0.1505 / 1e12)
    # one rank alone reproduces the single-GPU figure
    assert bench.replicas_tflops(1, flops, 10, 120.0) == pytest.approx(flops * 10 / 0.120 / 1e12)


def test_single_process_needs_no_group():
    assert bench.slowest_rank_ms(42.0) == 42.0


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 1, 0, 2
    bench.run_reference(Args())
    assert capsys.readouterr().out == ""
