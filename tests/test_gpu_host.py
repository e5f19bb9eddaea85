"""moe_ffn_forward_host: the forward pass from host memory in token chunks
whose copies in and out overlap the computation of the neighbouring chunks.
Every chunk is one forward call, so each output row is checked against the
oracle at the path's tolerances, for one chunk, several chunks with a ragged
last one, more chunks than staging sets (buffer reuse), pageable as well as
page-locked host memory, MXFP8, and a reported bad expert id."""
import numpy as np
import pytest
import torch

import grouped_gemm_gb300 as moe
import oracle
from grouped_gemm_gb300 import workloads as wl

from helpers import assert_close, coverage_tokens

pytestmark = pytest.mark.gpu


def host_inputs(inp, pinned=True):
    def h(a):
        t = torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a))
        return t.pin_memory() if pinned else t
    d = {key: h(inp[key]) for key in ("x", "topk_ids", "topk_w") if key in inp}
    if "x_sf" in inp:
        d["x_sf"] = h(inp["x_sf"])
    return d


def run_host(inp, chunk, pinned=True, pipeline=moe.MOE_SPLIT, dtype=moe.MOE_BF16, check=True):
    w = inp["workload"]
    T, D, H, E, k = w.T, w.D, w.H, w.E, w.k
    hb = host_inputs(inp, pinned)
    w1 = torch.from_numpy(inp["w1"].view(np.int16) if inp["w1"].dtype == np.uint16 else inp["w1"]).cuda()
    w2 = torch.from_numpy(inp["w2"].view(np.int16) if inp["w2"].dtype == np.uint16 else inp["w2"]).cuda()
    w1p = w2p = None
    if dtype != moe.MOE_BF16:
        w1p = torch.empty(inp["w1_sf"].size, dtype=torch.uint8, device="cuda")
        w2p = torch.empty(inp["w2_sf"].size, dtype=torch.uint8, device="cuda")
        moe.moe_ffn_prepare_mxfp8_weights(torch.from_numpy(inp["w1_sf"]).cuda(), torch.from_numpy(inp["w2_sf"]).cuda(),
                                          w1p, w2p, E, D, H)
    out = torch.full((T, D), float("nan"), dtype=torch.bfloat16)
    out = out.pin_memory() if pinned else out
    n = moe.moe_ffn_host_workspace_size(T, E, D, H, k, dtype, pipeline, chunk_tokens=chunk)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    moe.moe_ffn_workspace_init(ws)
    moe.moe_ffn_forward_host(hb["x"], w1, w2, hb["topk_ids"], hb["topk_w"], out, E=E, D=D, H=H, k=k, workspace=ws,
                             dtype=dtype, pipeline=pipeline, x_sf=hb.get("x_sf"), w1_sf=w1p, w2_sf=w2p,
                             chunk_tokens=chunk)
    torch.cuda.current_stream().synchronize()
    st = moe.moe_ffn_sync_status(ws)
    if check:
        assert st == 0, moe.moe_ffn_status_string(st)
    return out, st


def oracle_out(inp, dtype="bf16", tokens=None):
    if dtype == "mxfp8":
        return oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_MXFP8,
                              x_sf=inp["x_sf"], w1_sf=inp["w1_sf"], w2_sf=inp["w2_sf"], tokens=tokens)
    return oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_BF16,
                          tokens=tokens)


@pytest.mark.parametrize("pipeline", [moe.MOE_SPLIT, moe.MOE_FUSED])
@pytest.mark.parametrize("chunk", [0, 300, 64, 7])   # one chunk; one exact chunk; 5 with a ragged last; 43 chunks
def test_host_forward_chunks(chunk, pipeline):
    inp = wl.make_custom(300, 512, 256, 16, 4, seed=31, routing="uniform")
    out, _ = run_host(inp, chunk, pipeline=pipeline)
    assert_close(out, oracle_out(inp), label=f"host chunk={chunk}")


def test_host_forward_ramped_chunks():
    # eight chunks or more: a quarter chunk first and last ([128, 512 x 8, 256, 128] here)
    inp = wl.make_custom(4608, 256, 128, 8, 2, seed=35, routing="uniform")
    out, _ = run_host(inp, 512)
    assert_close(out, oracle_out(inp), label="host ramped chunks")


def test_host_forward_pageable_memory():
    inp = wl.make_custom(200, 256, 128, 8, 2, seed=32, routing="topk_logits")
    out, _ = run_host(inp, 48, pinned=False)
    assert_close(out, oracle_out(inp), label="host pageable")


def test_host_forward_mxfp8_chunks():
    inp = wl.make_custom(300, 512, 256, 16, 4, seed=33, routing="uniform", dtype="mxfp8")
    out, _ = run_host(inp, 128, dtype=moe.MOE_MXFP8)
    assert_close(out, oracle_out(inp, "mxfp8"), dtype="mxfp8", label="host mxfp8")


def test_host_forward_prefill_workload_sampled():
    # the prefill workload in four chunks; every expert's first, last and tail rows + 1000 random tokens
    inp = wl.make_inputs("prefill", seed=0)
    out, _ = run_host(inp, 1024)
    tokens = coverage_tokens(inp["topk_ids"], seed=3)
    assert_close(out[torch.from_numpy(tokens.astype(np.int64))], oracle_out(inp, tokens=tokens), label="host prefill")


def test_host_forward_reports_a_bad_expert_id():
    inp = wl.make_custom(200, 256, 128, 8, 2, seed=34, routing="uniform")
    inp["topk_ids"][150, 1] = 8                 # outside [0, E), in the third chunk of 64
    out, st = run_host(inp, 64, check=False)
    assert st == 4
    ids = inp["topk_ids"].copy()
    tw = inp["topk_w"].copy()
    ids[150, 1] = 0
    tw[150, 1] = 0.0
    ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], ids, tw, act=oracle.ACT_BF16)
    assert_close(out, ref, label="host bad id dropped")
