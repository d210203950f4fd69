"""The benchmark's multi-rank host logic under gloo on CPU, world size 2:
every rank draws its own batch, the step time is the slowest rank's, and the
job's throughput counts every rank's tokens (replicas, weak scaling)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import ssd_inputs as si


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        assert (r, lr, w) == (rank, rank, world)
        cfg = bench.rank_config(si.CONFIGS["tiny_f32"], rank)
        x = si.make_inputs(cfg).x
        ms = 1.0 + rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, world)
        out[rank] = (float(np.asarray(x, dtype=np.float64).sum()), slowest,
                     bench.job_tokens_per_s(cfg.tokens, world, slowest))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    (s0, m0, v0), (s1, m1, v1) = out[0], out[1]
    assert s0 != s1, "ranks drew the same batch"
    assert m0 == m1 == 2.0, "step time is not the slowest rank's"
    tokens = si.CONFIGS["tiny_f32"].tokens
    assert v0 == v1 == pytest.approx(world * tokens / 2e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_tokens_per_s(1000, 1, 1.0) == pytest.approx(1e6)


def test_clock_sampler_names_the_physical_gpu(monkeypatch):
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES", raising=False)
    assert bench.smi_gpu_id(0) == "0" and bench.smi_gpu_id(3) == "3"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "4,6")
    assert bench.smi_gpu_id(0) == "4" and bench.smi_gpu_id(1) == "6"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "GPU-abc, GPU-def")
    assert bench.smi_gpu_id(1) == "GPU-def"
