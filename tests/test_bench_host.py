"""Host-side helpers of bench.py (no GPU): the kernel each workload's step
takes (the roofline line names it), the algorithmic bytes per parameter,
and the rule that the recorded DRAM traffic is reported only for the kernel
sources it was taken on."""

import os

import pytest

import bench


@pytest.mark.parametrize("n,gd,keep,elems,want", [
    (8, "bf16", False, 73_417_728, "step_pipe_kernel"),       # the Llama-1024 workload
    (8, "bf16", False, 2 ** 23 - 1, "step_vec_kernel"),
    (1, "bf16", False, 2 ** 23, "step_tma4_kernel"),
    (2, "bf16", False, 10 ** 9, "step_tma4_kernel"),
    (4, "bf16", False, 10 ** 9, "step_tma4_kernel"),
    (5, "bf16", False, 10 ** 9, "step_vec_kernel"),
    (6, "bf16", False, 10 ** 9, "step_vec_kernel"),
    (7, "bf16", False, 10 ** 9, "step_pipe_kernel"),
    (10, "bf16", False, 10 ** 9, "step_pipe_kernel"),
    (12, "bf16", False, 10 ** 9, "step_pipe_kernel"),
    (13, "bf16", False, 10 ** 9, "step_tma_kernel"),
    (16, "bf16", False, 10 ** 9, "step_tma_kernel"),
    (16, "bf16", False, 10 ** 6, "step_vec_kernel"),          # small launches stay register-staged
    (2, "fp32", False, 2_030_174_208, "step_vec_kernel"),     # the stage-buffer workload
    (6, "fp32", False, 10 ** 9, "step_vec_kernel"),
    (7, "fp32", False, 10 ** 9, "step_tma4_kernel"),
    (8, "fp32", False, 10 ** 9, "step_tma_kernel"),
    (9, "fp32", False, 10 ** 9, "step_tma_kernel"),
    (10, "fp32", False, 10 ** 9, "step_tma4_kernel"),
    (16, "fp32", False, 10 ** 9, "step_tma4_kernel"),
    (16, "bf16", True, 10 ** 9, "step_vec_kernel"),           # kept reduced gradient: one fp32 replica
])
def test_step_kernel_name(n, gd, keep, elems, want):
    assert bench.step_kernel_name(n, gd, keep, elems) == want


def test_bytes_per_param():
    assert bench.bytes_per_param(8, "bf16") == 42
    assert bench.bytes_per_param(2, "fp32") == 34
    assert bench.bytes_per_param(1, "bf16") == 28


def test_workload_shapes():
    wl = bench.workload("llama1024_zero2_n8")
    assert (wl["n"], wl["stage"], wl["grad_dtype"]) == (8, 2, "bf16")
    assert sum(wl["pl"].numel) == 73_417_728
    wl = bench.workload("flat32:4e6:12")
    assert (wl["n"], wl["stage"], wl["grad_dtype"], sum(wl["pl"].numel)) == (12, 1, "fp32", 4_000_000)
    with pytest.raises(SystemExit):
        bench.workload("no_such_workload")


def test_traffic_only_for_the_recorded_sources(tmp_path, monkeypatch):
    sha = bench.kernel_source_sha()
    assert len(sha) == 16 and sha == bench.kernel_source_sha()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "step_kernel_dram_traffic.txt").write_text(
        "# comment\n"
        f"workload=w1 kernel_sha={sha} dram_bytes_per_launch=123\n"
        "workload=w2 kernel_sha=0000000000000000 dram_bytes_per_launch=456\n")
    # the sources are read from the real tree, the record from the temporary one
    real_root = bench.ROOT
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: sha)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("w1") == 123.0
    assert bench.recorded_traffic("w2") is None          # taken on other sources
    assert bench.recorded_traffic("w3") is None          # not recorded
    monkeypatch.setattr(bench, "ROOT", real_root)
    assert os.path.exists(os.path.join(real_root, "profiles", "step_kernel_dram_traffic.txt"))


def test_default_workload_is_the_stage_buffer():
    # the default line is the largest single-GPU workload: the 2.03 B-param
    # stage buffer, N = 2, ZeRO-1, fp32 gradients (34 B/param)
    assert bench.DEFAULT_WORKLOAD == "stage_buffer_zero1_fp32_n2"
    wl = bench.workload(bench.DEFAULT_WORKLOAD)
    assert (wl["n"], wl["stage"], wl["grad_dtype"], wl["pl"].total) == (2, 1, "fp32", 2_030_174_208)
    cfg = bench.config_for(bench.DEFAULT_WORKLOAD, wl, 1)
    assert cfg["params"] == 2_030_174_208 and cfg["units"] == 1 and cfg["n_ranks_simulated"] == 2
    assert cfg["l2"].startswith("inputs larger than L2: 69.03 GB")
    for name in bench.ALSO_WORKLOADS:
        bench.workload(name)


def test_config_is_a_function_of_the_workload_only():
    wl = bench.workload("llama2048_zero3_n8")
    a, b = bench.config_for("llama2048_zero3_n8", wl, 1), bench.config_for("llama2048_zero3_n8", wl, 1)
    assert a == b and a["units"] == 10 and a["zero_stage"] == 3
    assert bench.config_for("toy_mlp_n4", bench.workload("toy_mlp_n4"), 1)["l2"].startswith("working set fits L2")


def test_llama2048_workloads_at_other_rank_counts():
    wl = bench.workload("llama2048_zero3_n6_unitbufs")
    assert (wl["n"], wl["stage"], wl["unit_bufs"], wl["pl"].n_units) == (6, 3, True, 10)
    wl = bench.workload("llama2048_zero3_n3")
    assert (wl["n"], wl["unit_bufs"]) == (3, False)
    for bad in ("llama2048_zero3_n6_x", "llama2048_zero3_nx"):
        with pytest.raises(SystemExit):
            bench.workload(bad)
