"""Failure detection without a GPU fault: every wait inside the kernels is
bounded.  With the MOE_OPT_TEST_STALL hook the MMA issuer waits on a barrier
that nothing arrives on; with a 1 ms bound that wait runs out, the kernels
record MOE_ERR_DEVICE_TIMEOUT in the workspace status words and exit cleanly
(in-flight copies and MMAs drained, tensor memory freed), and the next call on
the same context is correct.  Bad expert ids are reported the same way."""
import numpy as np
import pytest
import torch

import grouped_gemm_gb300 as moe
import oracle
from grouped_gemm_gb300 import workloads as wl

from helpers import assert_close, run_forward, to_dev

pytestmark = pytest.mark.gpu


def oracle_out(inp):
    return oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_BF16)


# (pipeline, MOE_OPT_FUSED_CLUSTER, MOE_OPT_PAIR_MMA): split on single CTAs and
# on CTA pairs; fused on clusters of two CTAs (D = 512); fused with H-split
# fp32 partial sums
@pytest.mark.parametrize("pipeline,cluster,pair", [(moe.MOE_SPLIT, 1, 0), (moe.MOE_SPLIT, 1, 1),
                                                   (moe.MOE_FUSED, 1, 2), (moe.MOE_FUSED, 0, 2)])
def test_wait_timeout_is_reported_and_context_survives(pipeline, cluster, pair):
    inp = wl.make_custom(300, 512, 256, 16, 4, seed=3)
    dev = to_dev(inp)
    moe.moe_ffn_set_wait_limit_ns(1_000_000)
    moe.moe_ffn_set_option(moe.MOE_OPT_TEST_STALL, 1)
    moe.moe_ffn_set_option(moe.MOE_OPT_FUSED_CLUSTER, cluster)
    moe.moe_ffn_set_option(moe.MOE_OPT_PAIR_MMA, pair)
    try:
        _, ws = run_forward(inp, dev, pipeline=pipeline, check_status=False)
        st = moe.moe_ffn_sync_status(ws)
    finally:
        moe.moe_ffn_set_option(moe.MOE_OPT_TEST_STALL, 0)
        moe.moe_ffn_set_option(moe.MOE_OPT_FUSED_CLUSTER, 1)
        moe.moe_ffn_set_option(moe.MOE_OPT_PAIR_MMA, 2)
        moe.moe_ffn_set_wait_limit_ns(2_000_000_000)
    assert st == 6, moe.moe_ffn_status_string(st)
    assert moe.moe_ffn_sync_status(ws) == 0          # status words cleared by the read
    out, _ = run_forward(inp, dev, pipeline=pipeline, workspace=ws)
    assert_close(out, oracle_out(inp), label="after timeout")


def test_bad_expert_id_is_reported():
    inp = wl.make_custom(64, 256, 128, 8, 2, seed=4)
    inp["topk_ids"][7, 1] = 8                       # outside [0, E)
    dev = to_dev(inp)
    out, ws = run_forward(inp, dev, check_status=False)
    assert moe.moe_ffn_sync_status(ws) == 4
    # the pair is dropped; every other token is still computed correctly
    ids = inp["topk_ids"].copy()
    tw = inp["topk_w"].copy()
    ids[7, 1] = 0
    tw[7, 1] = 0.0
    ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], ids, tw, act=oracle.ACT_BF16)
    assert_close(out, ref, label="bad id dropped")


@pytest.mark.parametrize("pipeline", [moe.MOE_SPLIT, moe.MOE_FUSED])
def test_routing_barrier_timeout_is_reported_and_context_survives(pipeline):
    # 4000 tokens x 4 = 16000 pairs: the one-launch cooperative routing, whose
    # block 0 leaves before the first grid barrier (MOE_OPT_TEST_STALL 2)
    inp = wl.make_custom(4000, 256, 128, 16, 4, seed=8)
    dev = to_dev(inp)
    moe.moe_ffn_set_wait_limit_ns(1_000_000)
    moe.moe_ffn_set_option(moe.MOE_OPT_TEST_STALL, 2)
    try:
        out, ws = run_forward(inp, dev, pipeline=pipeline, check_status=False)
        st = moe.moe_ffn_sync_status(ws)
    finally:
        moe.moe_ffn_set_option(moe.MOE_OPT_TEST_STALL, 0)
        moe.moe_ffn_set_wait_limit_ns(2_000_000_000)
    assert st == 6, moe.moe_ffn_status_string(st)
    assert torch.isfinite(out.float()).all()        # zero-filled, no stale rows
    assert moe.moe_ffn_sync_status(ws) == 0
    out, _ = run_forward(inp, dev, pipeline=pipeline, workspace=ws)
    assert_close(out, oracle_out(inp), label="after routing timeout")
