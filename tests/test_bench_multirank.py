"""Host-side logic of bench.py's multi-rank (token-sharded, weak-scaling) path
on CPU with the gloo backend, world size 2: the step time is the slowest
rank's, the value aggregates every rank's work, and the reference arm runs on
rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = [2.0, 5.0][rank]
        ms = bench.max_over_ranks(ms_local, world)
        value = bench.weak_scaling_tflops(1e12, ms, world)
        dist.barrier()
        results[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        ms, value = results[r]
        assert ms == 5.0
        assert value == pytest.approx(1e12 * 2 / 5e-3 / 1e12)


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.weak_scaling_tflops(2e12, 1.0, 1) == pytest.approx(2000.0)


def test_reference_arm_only_on_rank0():
    class A:
        workload, steps, warmup, gpus, pipeline = "tiny", 1, 0, 2, "split"
    assert bench.run_reference(A(), rank=1) is None


def test_reference_arm_line_contract():
    # the CPU oracle as the reference arm: one JSON line with the same metric,
    # its own cpu_baseline and an e2e with no host-device traffic
    class A:
        workload, steps, warmup, gpus, pipeline = "tiny", 1, 0, 1, "split"
    line = bench.run_reference(A(), rank=0)
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "tiny"


def test_algorithmic_counts():
    import numpy as np
    from grouped_gemm_gb300 import workloads as wl
    w = wl.WORKLOADS["tiny"]
    ids = np.array([[0, 1]] * w.T, np.int32)          # two live experts
    alg = bench.algorithmic(w, ids)
    P = w.T * w.k
    assert alg["step_flops"] == 6.0 * P * w.D * w.H
    assert alg["up_swiglu"]["flops"] + alg["down_reduce"]["flops"] == alg["step_flops"]
    # compulsory bytes: x, the live experts' weights, ids and weights, out
    assert alg["step_bytes"] == w.T * w.D * 2 + 2 * 3 * w.H * w.D * 2 + P * 8 + w.T * w.D * 2
    assert alg["live_experts"] == 2


def test_gemm_only_figure():
    # split: up + down; fused: the fused GEMM and its rounding pass
    g = bench.gemm_only({"route": 0.02, "gather_zero": 0.03, "up_swiglu": 0.2, "down_reduce": 0.1}, "split", 3e11)
    assert g["ms"] == pytest.approx(0.3) and g["tflops"] == pytest.approx(3e11 / 0.3e-3 / 1e12)
    g = bench.gemm_only({"route": 0.02, "gather_zero": 0.03, "fused_gemm": 0.4, "to_bf16": 0.0}, "fused", 4e11)
    assert g["ms"] == pytest.approx(0.4) and g["stages"] == ["fused_gemm", "to_bf16"]
    assert bench.gemm_only({"route": 0.02}, "split", 1e9) is None


def test_host_cpu_record():
    h = bench.host_cpu()
    assert h["model"] and h["nproc"] >= 1 and h["omp_threads"] >= 1


def test_roofline_fractions_measured_and_nominal():
    import numpy as np
    from grouped_gemm_gb300 import workloads as wl
    w = wl.WORKLOADS["large_skewed"]
    ids = np.tile(np.arange(8, dtype=np.int32), (w.T, 1))
    alg = bench.algorithmic(w, ids)
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1800.0}
    stage_ms = {"route": 0.03, "gather_zero": 0.5, "up_swiglu": 4.0, "down_reduce": 2.0}
    kern = {"route": "route_coop", "gather_zero": "gather_tokens", "up_swiglu": "up_swiglu_pair2",
            "down_reduce": "down_reduce_pair2"}
    roof, step_bound, step_nom = bench.roofline_fracs(alg, stage_ms, "split", False, peaks, "measured", kern,
                                                      "large_skewed")
    # the up projection (the longer stage) is tensor-bound: FLOPs over its time
    achieved = alg["up_swiglu"]["flops"] / 4e-3 / 1e12
    assert roof["bound"] == "tensor" and roof["kernel"] == "up_swiglu_pair2"
    assert roof["frac"] == pytest.approx(achieved / 1800.0, rel=1e-3)
    assert roof["frac_nominal"] == pytest.approx(achieved / bench.NOMINAL_PEAKS["bf16_tflops"], rel=1e-3)
    assert step_bound == pytest.approx(alg["step_flops"] / 1.8e15)
    assert step_nom == pytest.approx(alg["step_flops"] / 2.25e15)
    # MXFP8: the fp8 peaks (twice the measured bf16 one; the data-sheet fp8 figure)
    roof8, sb8, sn8 = bench.roofline_fracs(alg, stage_ms, "split", True, peaks, "measured", kern, "mxfp8")
    assert roof8["peak"] == 3600.0 and roof8["peak_nominal"] == bench.NOMINAL_PEAKS["fp8_tflops"]


def test_clock_summary_keeps_samples_inside_the_window():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.source = "test"
    s.samples = [(1.0, 1500.0, 2070.0, []), (2.0, 2000.0, 2070.0, ["sw_power_cap"]), (2.5, 2070.0, 2070.0, []),
                 (4.0, 900.0, 2070.0, ["hw_slowdown"])]
    c = s.summary(1.5, 3.0)
    assert c["samples"] == 2 and c["sm_mhz"] == pytest.approx(2035.0) and c["reasons"] == ["sw_power_cap"]
    assert s.summary(5.0, 6.0) is None
