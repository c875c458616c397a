"""Host logic of bench.py for N > 1 ranks, on CPU with the gloo backend
(world size 2): the max-over-ranks time, the whole-job throughput, and the
reference arm running on rank 0 only.
"""

import contextlib
import io
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench._max_over_ranks(values[rank], world, "cpu")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        values = [3.25, 7.5]
        mp.start_processes(_rank_main, args=(2, _free_port(), values, out), nprocs=2,
                           start_method="spawn", join=True)
        assert dict(out) == {0: 7.5, 1: 7.5}


def test_max_over_ranks_single_rank_is_identity():
    assert bench._max_over_ranks(1.5, 1, "cpu") == 1.5


def test_whole_job_tflops_counts_every_rank():
    # 1e12 FLOPs per rank in 2 ms on each of 4 ranks: 4e12 FLOPs / 2 ms = 2000 TFLOP/s
    assert bench._whole_job_tflops(1e12, 4, 2.0) == pytest.approx(2000.0)
    assert bench._whole_job_tflops(1e12, 1, 2.0) == pytest.approx(500.0)


def test_reference_arm_runs_on_rank0_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.run_reference(None)      # a non-zero rank returns before reading args
    assert rc == 0 and buf.getvalue() == ""
