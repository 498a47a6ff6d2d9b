"""The benchmark's multi-rank path on CPU (not gpu): two gloo ranks on
127.0.0.1.  Every rank runs its own replica of the workload (no data-path
collective); the job's time is the max over ranks and its throughput the sum
of the units all ranks processed.  The reference arm runs on rank 0 only."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        bench.barrier(world)
        local_ms = 10.0 + 5.0 * rank          # rank 1 is slower
        local_params = 1000.0 * (rank + 1)
        mx = bench.aggregate([local_ms], "max", world, "cpu")[0]
        tot = bench.aggregate([local_params], "sum", world, "cpu")[0]
        out[rank] = (mx, tot)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1] == (15.0, 3000.0)


def _ref_worker(rank, world, out):
    import contextlib
    import io

    import bench
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))

    class Args:
        workload = "toy_mlp_n4"
        steps = 2
        warmup = 1
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(Args())
    out[rank] = buf.getvalue()


def test_reference_arm_runs_on_rank0_only():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_ref_worker, args=(2, out), nprocs=2, join=True, start_method="spawn")
    import json
    line = json.loads(out[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert out[1] == ""
    # the same config dict the GPU arm prints for this workload and launch
    import bench
    assert line["config"] == bench.config_for("toy_mlp_n4", bench.workload("toy_mlp_n4"), 2)
    assert (line["steps"], line["warmup"]) == (2, 1)
