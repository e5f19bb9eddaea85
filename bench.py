#!/usr/bin/env python
"""Benchmark of the routed MoE SwiGLU FFN forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload large_skewed]
                    [--pipeline split] [--impl ours|reference] [--no-also]

One step = one full forward pass (routing, gather + zero-fill, up-projection
with SwiGLU, down-projection with the weighted reduction) over one batch of
seeded synthetic inputs already resident in HBM.  The default workload is the
largest one (T=131072 tokens, D=2048, H=768, E=128, top-8, Zipf-skewed
routing) on the split pipeline.  Prints ONE JSON line on rank 0; at N=1 it
also carries, under "other_configs", the same measurement (timed steps,
per-stage kernel fractions, clocks) of the other workloads and pipelines,
taken in the same run after the main one.  Under torchrun each rank runs its own token batch against its own
copy of the weights (the path shards by tokens, no collective on the data
path): weak scaling, value = all ranks' FLOPs / max-over-ranks time.

--impl reference times the CPU oracle (fp64, OpenMP) on the host cores, on a
bounded sample of tokens per step, with the same metric and workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE FFN fwd TFLOP/s & tokens/s on 1×GB300; % of roofline (tensor or HBM)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 data-sheet figures (dense, no sparsity), reported beside the measured-peak fractions
NOMINAL_PEAKS = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0, "fp8_tflops": 4500.0, "fp4_tflops": 13500.0}
# measured after the main workload in the same run (N=1): workload, pipeline
ALSO = [("large_skewed", "split"), ("large_skewed", "fused"), ("prefill", "split"), ("prefill", "fused"),
        ("mxfp8", "split"), ("mxfp8", "fused"), ("decode", "split"), ("decode", "fused"),
        ("decode_mxfp4w", "split"), ("decode_nvfp4", "split")]
STAGES = {"split": ["route", "gather_zero", "up_swiglu", "down_reduce"],
          "fused": ["route", "gather_zero", "fused_gemm", "to_bf16"]}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="large_skewed")
    ap.add_argument("--pipeline", choices=["split", "fused"], default="split")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--from-logits", action="store_true",
                    help="start each step from router logits [T, E] (moe_ffn_forward_logits: top-k and softmax "
                         "fused into the routing launch) instead of given top-k ids and weights")
    ap.add_argument("--no-graph", action="store_true", help="launch each step eagerly instead of replaying a CUDA graph")
    ap.add_argument("--host-chunk", type=int, default=0,
                    help="e2e: token chunk of the host-buffer entry point (0: the library's automatic choice)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count T (a smaller case of the same kernels, for profiling)")
    ap.add_argument("--no-also", action="store_true",
                    help="skip the other workloads and pipelines measured after the main one (N=1 only)")
    ap.add_argument("--option", action="append", default=[], metavar="NAME=VALUE",
                    help="library tuning option, e.g. PAIR_MMA=0 (moe_ffn_set_option; repeatable)")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def algorithmic(w, ids):
    """Compulsory bytes and FLOPs of the whole step and of each GEMM kernel."""
    import numpy as np
    P = w.T * w.k
    live = int(np.unique(ids).size)
    eb = 2 if w.dtype == "bf16" else 0.5 if w.dtype == "nvfp4" else 1
    sfb = 0 if w.dtype == "bf16" else 1.0 / 16 if w.dtype == "nvfp4" else 1.0 / 32
    elem = eb + sfb                                              # activations (x, act)
    welem = (0.5 + sfb) if w.dtype == "mxfp4w" else elem         # expert weights
    step_bytes = (w.T * w.D * elem + live * 3 * w.H * w.D * welem + P * 8 + w.T * w.D * 2)
    up_bytes = live * 2 * w.H * w.D * welem + P * w.D * elem + P * w.H * elem
    down_bytes = live * w.D * w.H * welem + P * w.H * elem + w.T * w.D * 2
    return {
        "step_flops": 6.0 * P * w.D * w.H, "step_bytes": float(step_bytes),
        "up_swiglu": {"flops": 4.0 * P * w.D * w.H, "bytes": float(up_bytes)},
        "down_reduce": {"flops": 2.0 * P * w.D * w.H, "bytes": float(down_bytes)},
        "live_experts": live,
    }


def gemm_only(stage_ms, pipeline, step_flops):
    """The GEMM stages alone (routing and gather excluded, as in the pages'
    timed region): their summed per-stage durations and the step's FLOPs over
    that time.  None when a stage is missing."""
    names = ["up_swiglu", "down_reduce"] if pipeline == "split" else ["fused_gemm", "to_bf16"]
    if any(n not in stage_ms for n in names):
        return None
    ms = sum(stage_ms[n] for n in names)
    if ms <= 0:
        return None
    return {"ms": round(ms, 5), "tflops": round(step_flops / (ms * 1e-3) / 1e12, 3), "stages": names}


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


_PTX = ["grouped_gemm_gb300/csrc/ptx.cuh", "grouped_gemm_gb300/csrc/internal.h"]
_MXH = ["grouped_gemm_gb300/csrc/mx.cuh"]
# kernel name (moe_ffn_profile_stage_kernel) -> the sources it is built from
KERNEL_SOURCES = {
    "up_swiglu_bf16": ["grouped_gemm_gb300/csrc/gemm_bf16.cu"] + _PTX,
    "down_reduce_bf16": ["grouped_gemm_gb300/csrc/gemm_bf16.cu"] + _PTX,
    "up_swiglu_pair2": ["grouped_gemm_gb300/csrc/gemm_pair2.cu"] + _PTX,
    "down_reduce_pair2": ["grouped_gemm_gb300/csrc/gemm_pair2.cu"] + _PTX,
    "up_swiglu_pair2_wide": ["grouped_gemm_gb300/csrc/gemm_pair2_wide.cu"] + _PTX,
    "up_swiglu_bf16_m64": ["grouped_gemm_gb300/csrc/gemm_bf16.cu"] + _PTX,
    "down_reduce_bf16_m64": ["grouped_gemm_gb300/csrc/gemm_bf16.cu"] + _PTX,
    "up_pair_bf16": ["grouped_gemm_gb300/csrc/gemm_pair.cu"] + _PTX,
    "up_swiglu_mxfp8": ["grouped_gemm_gb300/csrc/gemm_mxfp8.cu"] + _MXH + _PTX,
    "down_reduce_mxfp8": ["grouped_gemm_gb300/csrc/gemm_mxfp8.cu"] + _MXH + _PTX,
    "up_swiglu_mxfp8_pair2": ["grouped_gemm_gb300/csrc/gemm_mxfp8_pair.cu"] + _MXH + _PTX,
    "up_swiglu_mxfp8_swap": ["grouped_gemm_gb300/csrc/gemm_mx_swap.cu", "grouped_gemm_gb300/csrc/mx_swap.h"] + _MXH + _PTX,
    "down_reduce_mxfp8_swap": ["grouped_gemm_gb300/csrc/gemm_mx_swap.cu", "grouped_gemm_gb300/csrc/mx_swap.h"] + _MXH + _PTX,
    "up_swiglu_mxfp4w_swap": ["grouped_gemm_gb300/csrc/gemm_mx_swap.cu", "grouped_gemm_gb300/csrc/mx_swap.h"] + _MXH + _PTX,
    "down_reduce_mxfp4w_swap": ["grouped_gemm_gb300/csrc/gemm_mx_swap.cu", "grouped_gemm_gb300/csrc/mx_swap.h"] + _MXH + _PTX,
    "down_reduce_mxfp8_pair2": ["grouped_gemm_gb300/csrc/gemm_mxfp8_pair.cu"] + _MXH + _PTX,
    "up_swiglu_mxfp4w": ["grouped_gemm_gb300/csrc/gemm_mxfp8.cu"] + _MXH + _PTX,
    "up_swiglu_nvfp4": ["grouped_gemm_gb300/csrc/gemm_nvfp4.cu"] + _MXH + _PTX,
    "down_reduce_nvfp4": ["grouped_gemm_gb300/csrc/gemm_nvfp4.cu"] + _MXH + _PTX,
    "down_reduce_mxfp4w": ["grouped_gemm_gb300/csrc/gemm_mxfp8.cu"] + _MXH + _PTX,
    "fused_cluster_bf16": ["grouped_gemm_gb300/csrc/gemm_fused_cluster.cu"] + _PTX,
    "fused_dsmem_bf16": ["grouped_gemm_gb300/csrc/gemm_fused_dsmem.cu"] + _PTX,
    "fused_moe_bf16": ["grouped_gemm_gb300/csrc/gemm_fused.cu"] + _PTX,
    "fused_cluster_mxfp8": ["grouped_gemm_gb300/csrc/gemm_fused_cluster_mx.cu"] + _MXH + _PTX,
    "fused_moe_mxfp8": ["grouped_gemm_gb300/csrc/gemm_fused_mx.cu"] + _MXH + _PTX,
    "route": ["grouped_gemm_gb300/csrc/route.cu"] + _PTX,
    "gather_tokens": ["grouped_gemm_gb300/csrc/route.cu"] + _PTX,
}


def traffic_from_profiles(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    sources are unchanged since the capture; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    d = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    if not m or not d or d.group(1) != source_digest(KERNEL_SOURCES.get(kernel, [])):
        return None
    return float(m.group(1))


class ClockSampler:
    """SM clock and clock-event reasons sampled every few milliseconds by a
    background thread through NVML (libnvidia-ml, read-only queries), so that
    even a timed region of a fraction of a second holds samples; nvidia-smi
    at 100 ms when NVML cannot be loaded."""
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    # NVML clock-event reason bits of those four
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index, period_s=0.005):
        self.samples = []        # (time, sm_mhz, sm_max_mhz, [reason names])
        self.proc = None
        self._stop = threading.Event()
        self.source = None
        if self._start_nvml(device_index, period_s):
            self.source = f"nvml every {period_s * 1e3:.0f} ms"
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.source = "nvidia-smi every 100 ms"
        self.thread = threading.Thread(target=self._read_smi, daemon=True)
        self.thread.start()

    def _start_nvml(self, device_index, period_s):
        import ctypes
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return False
            handle = ctypes.c_void_p()
            uuid = None
            try:
                import torch
                u = getattr(torch.cuda.get_device_properties(device_index), "uuid", None)
                uuid = f"GPU-{u}" if u is not None else None
            except Exception:
                uuid = None
            if not uuid or nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(handle)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(int(device_index), ctypes.byref(handle)) != 0:
                    return False
            clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            if nv.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) != 0:   # NVML_CLOCK_SM
                return False
        except (OSError, AttributeError):
            return False

        def loop():
            while not self._stop.is_set():
                ok = nv.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) == 0
                ok = ok and nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0
                ok = ok and reasons_fn(handle, ctypes.byref(rs)) == 0
                if ok:
                    names = [n for n, b in self.BITS.items() if rs.value & b]
                    self.samples.append((time.time(), float(clk.value), float(mx.value), names))
                time.sleep(period_s)

        self.thread = threading.Thread(target=loop, daemon=True)
        self.thread.start()
        return True

    def _read_smi(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                names = [self.NAMES[i] for i, v in enumerate(parts[5:9]) if v.lower() == "active"]
                self.samples.append((time.time(), float(parts[1]), float(parts[2]), names))
            except ValueError:
                pass

    def stop(self):
        self._stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for s in list(self.samples) if t0 <= s[0] <= t1]
        if not inside:
            return None
        sm = [s[1] for s in inside]
        reasons = sorted({n for s in inside for n in s[3]})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside), "source": self.source}


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (the slowest rank sets the step time)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_tflops(flops_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job throughput: every rank's FLOPs over the slowest rank's time."""
    return flops_per_rank * world / (ms_max * 1e-3) / 1e12


# ---------------------------------------------------------------- our arm
def roofline_fracs(alg, stage_ms, pipeline, mx, peaks, peak_src, stage_kernels, workload, fp4=False):
    """The dominant kernel's achieved rate against its roofline (measured
    peak, and the data-sheet peak beside it), and the step's bound."""
    if fp4:  # e2m1 x e2m1 contraction: the measured bf16 peak times the nominal fp4/bf16 ratio (13.5 / 2.25)
        peaks = dict(peaks)
        peaks["bf16_tflops"] = peaks["bf16_tflops"] * 6.0
        peak_src += " bf16 x nominal fp4/bf16 ratio 6"
    elif mx:  # e4m3 contraction: the measured bf16 peak times the nominal fp8/bf16 ratio (4.5 / 2.25)
        peaks = dict(peaks)
        peaks["bf16_tflops"] = peaks["bf16_tflops"] * 2.0
        peak_src += " bf16 x nominal fp8/bf16 ratio 2"
    nominal_tf = (NOMINAL_PEAKS["fp4_tflops"] if fp4 else NOMINAL_PEAKS["fp8_tflops"] if mx
                  else NOMINAL_PEAKS["bf16_tflops"])
    if pipeline == "split":
        dom = max(("up_swiglu", "down_reduce"), key=lambda s: stage_ms.get(s, 0.0))
        kd = alg[dom]
    else:
        dom = "fused_gemm"
        kd = {"flops": alg["up_swiglu"]["flops"] + alg["down_reduce"]["flops"], "bytes": alg["step_bytes"]}
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    tensor_bound = kd["flops"] / kd["bytes"] > ridge
    t_dom = stage_ms[dom] * 1e-3
    if tensor_bound:
        achieved, peak, nominal, unit = kd["flops"] / t_dom / 1e12, peaks["bf16_tflops"], nominal_tf, "TFLOP/s"
    else:
        achieved, peak, nominal, unit = kd["bytes"] / t_dom / 1e9, peaks["hbm_gbs"], NOMINAL_PEAKS["hbm_gbs"], "GB/s"
    kname = stage_kernels[dom]
    roofline = {"bound": "tensor" if tensor_bound else "hbm", "kernel": kname, "achieved": round(achieved, 1),
                "peak": peak, "peak_source": peak_src, "unit": unit, "frac": round(achieved / peak, 4),
                "peak_nominal": nominal, "frac_nominal": round(achieved / nominal, 4),
                "traffic": traffic_from_profiles(kname, workload),
                "algorithmic_per_launch": kd["flops"] if tensor_bound else kd["bytes"],
                "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()}, "stage_kernels": stage_kernels}
    step_bound = max(alg["step_flops"] / (peaks["bf16_tflops"] * 1e12), alg["step_bytes"] / (peaks["hbm_gbs"] * 1e9))
    step_bound_nominal = max(alg["step_flops"] / (nominal_tf * 1e12),
                             alg["step_bytes"] / (NOMINAL_PEAKS["hbm_gbs"] * 1e9))
    return roofline, step_bound, step_bound_nominal


def bench_workload(args, name, pipeline_name, rank, world, sampler, full=True):
    """Time one workload and pipeline (CUDA-graph replay of one step, inputs
    resident in HBM).  full: also the median of single replays, the clocks of
    a sustained run, the end-to-end pass from host buffers and the CPU
    baseline (the main line); otherwise the timed steps and the per-stage
    kernel fractions only (the other configurations of the same run)."""
    import numpy as np
    import torch

    import grouped_gemm_gb300 as moe
    from grouped_gemm_gb300 import workloads as wl

    inp = wl.make_inputs(name, seed=rank, T=args.tokens if name == args.workload else None)
    w = inp["workload"]
    nv = w.dtype == "nvfp4"                  # NVFP4 activations and weights, global scales
    mx = w.dtype in ("mxfp8", "mxfp4w", "nvfp4")  # block-scaled (one-byte or packed four-bit codes)
    dtype = {"bf16": moe.MOE_BF16, "mxfp8": moe.MOE_MXFP8, "mxfp4w": moe.MOE_MXFP4W, "nvfp4": moe.MOE_NVFP4}[w.dtype]
    dev = {k: torch.from_numpy(inp[k] if mx else inp[k].view(np.int16)).cuda() for k in ("x", "w1", "w2")}
    if nv:  # weight scales repacked once; the global scales as device scalars and vectors
        dev["x_sf"] = torch.from_numpy(inp["x_sf"]).cuda()
        dev["w1_sf"] = torch.empty(inp["w1_sf"].size, dtype=torch.uint8, device="cuda")
        dev["w2_sf"] = torch.empty(inp["w2_sf"].size, dtype=torch.uint8, device="cuda")
        moe.moe_ffn_prepare_nvfp4_weights(torch.from_numpy(inp["w1_sf"]).cuda(), torch.from_numpy(inp["w2_sf"]).cuda(),
                                          dev["w1_sf"], dev["w2_sf"], w.E, w.D, w.H)
        gs = {"x_gs": torch.tensor([float(inp["x_gs"])], dtype=torch.float32, device="cuda"),
              "w1_gs": torch.from_numpy(inp["w1_gs"]).cuda(), "w2_gs": torch.from_numpy(inp["w2_gs"]).cuda(),
              "act_gs": torch.tensor([float(inp["act_gs"])], dtype=torch.float32, device="cuda")}
    elif mx:  # weight scales are repacked once, like the weights themselves
        dev["x_sf"] = torch.from_numpy(inp["x_sf"]).cuda()
        dev["w1_sf"] = torch.empty(inp["w1_sf"].size, dtype=torch.uint8, device="cuda")
        dev["w2_sf"] = torch.empty(inp["w2_sf"].size, dtype=torch.uint8, device="cuda")
        moe.moe_ffn_prepare_mxfp8_weights(torch.from_numpy(inp["w1_sf"]).cuda(), torch.from_numpy(inp["w2_sf"]).cuda(),
                                          dev["w1_sf"], dev["w2_sf"], w.E, w.D, w.H)
    ids = torch.from_numpy(inp["topk_ids"]).cuda()
    tw = torch.from_numpy(inp["topk_w"]).cuda()
    logits = None
    if args.from_logits:  # the router's input; ids and weights become the call's outputs
        logits_np = wl.router_logits(w.T, w.E, seed=1000 + rank)
        logits = torch.from_numpy(logits_np).cuda()
    out = torch.empty(w.T, w.D, dtype=torch.bfloat16, device="cuda")
    pipeline = moe.MOE_SPLIT if pipeline_name == "split" else moe.MOE_FUSED
    ws = moe.alloc_workspace(w.T, w.E, w.D, w.H, w.k, dtype, pipeline)
    stream = torch.cuda.current_stream()

    def step():  # one forward pass on the current stream
        if nv:
            moe.moe_ffn_forward_nvfp4(dev["x"], dev["x_sf"], dev["w1"], dev["w1_sf"], dev["w2"], dev["w2_sf"],
                                      gs["x_gs"], gs["w1_gs"], gs["w2_gs"], gs["act_gs"], ids, tw, out, E=w.E, D=w.D,
                                      H=w.H, k=w.k, workspace=ws)
            return
        if logits is not None:
            moe.moe_ffn_forward_logits(dev["x"], dev["w1"], dev["w2"], logits, ids, tw, out, E=w.E, D=w.D, H=w.H,
                                       k=w.k, workspace=ws, dtype=dtype, pipeline=pipeline, x_sf=dev.get("x_sf"),
                                       w1_sf=dev.get("w1_sf"), w2_sf=dev.get("w2_sf"))
            return
        moe.moe_ffn_forward(dev["x"], dev["w1"], dev["w2"], ids, tw, out, E=w.E, D=w.D, H=w.H, k=w.k,
                            workspace=ws, dtype=dtype, pipeline=pipeline, x_sf=dev.get("x_sf"),
                            w1_sf=dev.get("w1_sf"), w2_sf=dev.get("w2_sf"))

    graph = None
    if not args.no_graph:
        # the pages time CUDA-graph replays; capture one step (after an eager
        # warm-up on a side stream, as torch requires)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
    timed_step = graph.replay if graph is not None else step

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(max(args.warmup, 3)):
        timed_step()
    torch.cuda.synchronize()
    st = moe.moe_ffn_sync_status(ws)
    if st != 0:
        raise SystemExit(f"device status after warm-up: {moe.moe_ffn_status_string(st)}")
    if logits is not None:  # the experts the router picked set the algorithmic bytes
        inp["topk_ids"] = ids.cpu().numpy()

    time.sleep(0.05)
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        timed_step()
    ev1.record(stream)
    ev1.synchronize()
    t_host1 = time.time()
    torch.cuda.synchronize()
    barrier()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world, device="cuda")
    ms = ms_total / args.steps
    t_sus0 = t_sus1 = None
    ms_median = None
    if full:
        # keep the same step running for 1.5 s: clocks under sustained load
        t_sus0 = time.time()
        while time.time() - t_sus0 < 1.5:
            for _ in range(20):
                timed_step()
            torch.cuda.synchronize()
        t_sus1 = time.time()
        # the pages' statistic beside the contract's mean: the median of single
        # replays, each between its own pair of events (a separate pass)
        n_med = max(1, min(args.steps, 50))
        med_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_med)]
        for i in range(n_med):
            med_ev[2 * i].record(stream)
            timed_step()
            med_ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        ms_median = max_over_ranks(
            statistics.median(med_ev[2 * i].elapsed_time(med_ev[2 * i + 1]) for i in range(n_med)), world,
            device="cuda")
    st = moe.moe_ffn_sync_status(ws)
    if st != 0:
        raise SystemExit(f"device status after timing: {moe.moe_ffn_status_string(st)}")

    alg = algorithmic(w, inp["topk_ids"])
    flops_all = alg["step_flops"] * world
    value = weak_scaling_tflops(alg["step_flops"], ms, world)
    tokens_per_s = w.T * world / (ms * 1e-3)

    # per-stage durations from library-recorded CUDA events on the same stream
    moe.moe_ffn_profile_enable(True)
    per = []
    for _ in range(min(args.steps, 30)):
        step()
        per.append(moe.moe_ffn_profile_read())
    names = STAGES[pipeline_name]
    stage_kernels = {nm: moe.moe_ffn_profile_stage_kernel(i) for i, nm in enumerate(names)}
    moe.moe_ffn_profile_enable(False)
    stage_ms = {nm: statistics.median(p[i] for p in per) for i, nm in enumerate(names) if len(per[0]) > i}
    # our kernels per step, from the kernels each stage launched ("a+b" = two)
    launches_per_step = sum(len(n.split("+")) for n in stage_kernels.values() if n and n != "none")

    peaks, peak_src = load_peaks()
    roofline, step_bound, step_bound_nominal = roofline_fracs(alg, stage_ms, pipeline_name, mx, peaks, peak_src,
                                                              stage_kernels, name, fp4=nv)
    clocks = sampler.summary(t_host0, t_host1) if sampler else None
    config = {"workload": w.name, "T": w.T, "D": w.D, "H": w.H, "E": w.E, "k": w.k, "routing": w.routing,
              "pipeline": pipeline_name, "seed": "rank", "parallelism": f"token-sharded x{world}",
              "options": args.option,
              "routing_input": "router logits [T, E] fp32" if args.from_logits else "top-k ids and weights",
              "launch": "eager" if graph is None else "CUDA graph replay of one step",
              "l2": (f"inputs larger than L2: {alg['step_bytes'] / 1e9:.2f} GB compulsory per step "
                     f"(129 MB L2), no flush needed")}
    line = {
        "value": round(value, 3), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
        "dtype": {"bf16": "bf16", "mxfp8": "e4m3 (MXFP8)", "mxfp4w": "e4m3 x e2m1 (MXFP8 x MXFP4)",
                  "nvfp4": "e2m1 (NVFP4)"}[w.dtype],
        "tokens_per_s": round(tokens_per_s, 1),
        "roofline_step_frac": round(step_bound / (ms * 1e-3), 4),
        "roofline_step_frac_nominal": round(step_bound_nominal / (ms * 1e-3), 4),
        "config": config, "roofline": roofline,
        "gemm_only": gemm_only(stage_ms, pipeline_name, alg["step_flops"]),
        "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
    }
    if not full:
        return line
    line["ms_per_step_median"] = round(ms_median, 5)
    if sampler:
        sus = sampler.summary(t_sus0, t_sus1)
        if sus is not None:
            sus["window"] = "the same step run for 1.5 s right after the timed region"
        line["clocks_sustained"] = sus

    # end to end: host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        xh = torch.from_numpy(inp["x"] if mx else inp["x"].view(np.int16)).pin_memory()
        xsfh = torch.from_numpy(inp["x_sf"]).pin_memory() if mx else None
        idh = torch.from_numpy(inp["topk_ids"]).pin_memory()
        twh = torch.from_numpy(inp["topk_w"]).pin_memory()
        lgh = torch.from_numpy(logits_np).pin_memory() if logits is not None else None
        outh = torch.empty(w.T, w.D, dtype=torch.bfloat16).pin_memory()
        # the host-buffer entry point (copies of one token chunk overlap the
        # computation of the neighbouring chunks) where it applies; router
        # logits and NVFP4: copies in, the step, the copy out, one after another
        host_api = logits is None and not nv
        if host_api:
            hws = torch.empty(moe.moe_ffn_host_workspace_size(w.T, w.E, w.D, w.H, w.k, dtype, pipeline,
                                                              chunk_tokens=args.host_chunk),
                              dtype=torch.uint8, device="cuda")
            moe.moe_ffn_workspace_init(hws)

        def e2e_step():
            if host_api:
                moe.moe_ffn_forward_host(xh, dev["w1"], dev["w2"], idh, twh, outh, E=w.E, D=w.D, H=w.H, k=w.k,
                                         workspace=hws, dtype=dtype, pipeline=pipeline, x_sf=xsfh,
                                         w1_sf=dev.get("w1_sf"), w2_sf=dev.get("w2_sf"), chunk_tokens=args.host_chunk)
                return
            dev["x"].copy_(xh, non_blocking=True)
            if mx:
                dev["x_sf"].copy_(xsfh, non_blocking=True)
            if logits is not None:
                logits.copy_(lgh, non_blocking=True)
            else:
                ids.copy_(idh, non_blocking=True)
                tw.copy_(twh, non_blocking=True)
            step()
            outh.copy_(out, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        n_e2e = max(1, min(args.steps, 100))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        e1.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world, device="cuda")
        e2e = {"value": round(flops_all / (e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(xh.numel() * xh.element_size() + (xsfh.numel() if mx else 0) +
                                         (lgh.numel() * 4 if logits is not None else idh.numel() * 4 + twh.numel() * 4)),
               "d2h_bytes_per_step": int(outh.numel() * 2), "ms_per_step": round(e_ms, 4),
               "resident": "expert weights stay in HBM (model parameters)",
               "call": (f"moe_ffn_forward_host (token chunks: {args.host_chunk or 'automatic'}; copies overlap "
                        "the neighbouring chunks' computation)" if host_api else
                        "copies in, the forward call, the copy out")}
        if host_api:
            st = moe.moe_ffn_sync_status(hws)
            if st != 0:
                raise SystemExit(f"device status after the host-buffer calls: {moe.moe_ffn_status_string(st)}")
    line["e2e"] = e2e
    line["cpu_baseline"] = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, w, budget_s=12.0)
    return line


def run_ours(args, rank, world, local_rank):
    import torch

    import grouped_gemm_gb300 as moe

    torch.cuda.set_device(local_rank)
    for opt in args.option:
        nm, val = opt.split("=")
        moe.moe_ffn_set_option(getattr(moe, "MOE_OPT_" + nm.upper()), int(val))
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    try:
        main = bench_workload(args, args.workload, args.pipeline, rank, world, sampler, full=True)
        torch.cuda.empty_cache()
        others = []
        if world == 1 and not args.no_also and not args.from_logits and not args.option and args.tokens is None:
            for name, pipe in ALSO:
                if (name, pipe) == (args.workload, args.pipeline):
                    continue
                try:
                    others.append(bench_workload(args, name, pipe, rank, world, sampler, full=False))
                except (RuntimeError, SystemExit, ValueError) as exc:   # one failing config does not lose the line
                    others.append({"config": {"workload": name, "pipeline": pipe}, "error": str(exc)[:300]})
                torch.cuda.empty_cache()
    finally:
        if sampler:
            sampler.stop()
    if rank != 0:
        return None
    line = {"metric": METRIC, "value": main["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "ms_per_step_median": main["ms_per_step_median"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": main["dtype"],
            "data": "synthetic"}
    for key in ("tokens_per_s", "roofline_step_frac", "roofline_step_frac_nominal", "config", "roofline",
                "cpu_baseline", "e2e", "gemm_only", "gpu_launches", "clocks", "clocks_sustained"):
        line[key] = main.get(key)
    if others:
        line["other_configs"] = others
    return line


def oracle_call(inp, tokens):
    import oracle
    dt = inp["workload"].dtype
    if dt == "nvfp4":
        return oracle.moe_ffn_nvfp4(inp["x"], inp["x_sf"], float(inp["x_gs"]), inp["w1"], inp["w1_sf"], inp["w1_gs"],
                                    inp["w2"], inp["w2_sf"], inp["w2_gs"], inp["topk_ids"], inp["topk_w"],
                                    act=oracle.ACT_NVFP4, act_gs=float(inp["act_gs"]), tokens=tokens)
    return oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"],
                          act=oracle.ACT_BF16 if dt == "bf16" else oracle.ACT_MXFP8, tokens=tokens,
                          x_sf=inp.get("x_sf"), w1_sf=inp.get("w1_sf"), w2_sf=inp.get("w2_sf"),
                          fp4_weights=dt == "mxfp4w")


def host_cpu():
    """The host's CPU model (lscpu), its logical CPU count and the oracle's
    OpenMP threads, for the CPU baseline's record."""
    import oracle
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"model": model or os.uname().machine, "nproc": os.cpu_count(), "omp_threads": oracle.max_threads()}


def cpu_baseline(inp, w, budget_s=12.0):
    """The oracle, as it stands, on the host cores over a bounded token sample."""
    import numpy as np

    import oracle
    per_tok = 6.0 * w.k * w.D * w.H
    n = 1
    t0 = time.time()
    oracle_call(inp, np.arange(n, dtype=np.int32))
    t1 = max(time.time() - t0, 1e-3)
    cores = oracle.max_threads()
    n = int(min(w.T, max(cores, budget_s / t1 * 0.9)))
    n = max(1, n // cores * cores) if n >= cores else n
    toks = np.sort(np.random.default_rng(123).choice(w.T, n, replace=False)).astype(np.int32)
    t0 = time.time()
    oracle_call(inp, toks)
    dt = time.time() - t0
    return {"value": round(per_tok * n / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {w.T} tokens of the {w.name} workload (all k={w.k} experts each), {dt:.1f} s",
            "tokens_per_s": round(n / dt, 3), "host": host_cpu()}


# ---------------------------------------------------------------- reference arm
def run_reference(args, rank):
    if rank != 0:
        return None
    import numpy as np

    import oracle
    from grouped_gemm_gb300 import workloads as wl
    inp = wl.make_inputs(args.workload, seed=0)
    w = inp["workload"]
    cores = oracle.max_threads()
    per_tok = 6.0 * w.k * w.D * w.H
    # tokens per step: about one second of CPU work
    t0 = time.time()
    oracle_call(inp, np.arange(min(cores, w.T), dtype=np.int32))
    t_one = max(time.time() - t0, 1e-3)
    n = int(max(1, min(w.T, min(cores, w.T) * max(1.0, 1.0 / t_one))))
    order = np.random.default_rng(7).permutation(w.T).astype(np.int32)

    def step(i):
        toks = np.sort(np.take(order, np.arange(i * n, (i + 1) * n) % w.T))
        oracle_call(inp, toks)

    for i in range(args.warmup):
        step(i)
    t0 = time.time()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.time() - t0
    ms = dt * 1e3 / args.steps
    value = per_tok * n / (ms * 1e-3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "D": w.D, "H": w.H, "E": w.E, "k": w.k, "routing": w.routing,
                   "pipeline": args.pipeline, "seed": 0, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} tokens of the {w.name} workload per step (all k={w.k} experts each)",
                         "host": host_cpu()},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank)
    else:
        if world > 1:
            import torch
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group(backend="nccl", device_id=torch.device("cuda", local_rank))
        line = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if line is not None and rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
