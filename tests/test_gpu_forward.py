"""End-to-end parity of the CUDA forward pass against the fp64 CPU oracle.

Tolerances: max|gpu - oracle| <= 2e-2 * max|oracle| and
sum|gpu - oracle| / sum|oracle| <= 5e-3 for bf16.  The oracle rounds act to
bf16 as the method does ("Prime Flash MoE" sec. 5, "SwiGLU - which never
leaves the SM").  Small cases are compared element by element over every
token; full-size workloads on a sample of tokens that reaches every expert's
first, last and tail rows plus seeded random tokens (outputs are independent
per token)."""
import numpy as np
import pytest
import torch

import grouped_gemm_gb300 as moe
import oracle
from grouped_gemm_gb300 import workloads as wl

from helpers import assert_close, cached_inputs, coverage_tokens, run_forward, to_dev

pytestmark = pytest.mark.gpu

# Pipeline and option settings under test: the split pipeline with the
# materializing gather kernel (default), with in-kernel gathers, with two row
# blocks per up tile, with the tail row blocks run as swap-AB tiles and with
# both GEMMs on CTA pairs (down tiles never swap-AB by default, or swap-AB for
# small pairs, or always; the up projection in 512-column tiles); the
# single-CTA GEMMs with 64-row tiles; the
# fused pipeline on clusters (default where the shape allows; act through the
# L2 ring, or kept in shared memory) and with the H-split fp32 partial sums.
MODES = {
    "split": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 0, moe.MOE_OPT_TILE_M: 128}),
    "split_pairs": (moe.MOE_SPLIT, {moe.MOE_OPT_UP_PAIRS: 1}),
    "split_gather4": (moe.MOE_SPLIT, {moe.MOE_OPT_GATHER: 1}),
    "split_cpasync": (moe.MOE_SPLIT, {moe.MOE_OPT_GATHER: 2}),
    "split_swap": (moe.MOE_SPLIT, {moe.MOE_OPT_SWAP_AB: 1}),
    "split_pair2": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 1}),
    "split_pair2_swap": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 1, moe.MOE_OPT_PAIR_SWAP: 128}),
    "split_pair2_allswap": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 1, moe.MOE_OPT_PAIR_SWAP: 256}),
    "split_pair2_half128": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 1, moe.MOE_OPT_HALF_PAIR_M128: 1}),
    "split_pair2_bands": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 1, moe.MOE_OPT_DOWN_BANDS: 3}),
    "split_pair2_epi4": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 1, moe.MOE_OPT_DOWN_EPI8: 0}),
    "split_pair2_noswap": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 1, moe.MOE_OPT_UP_SWAP: 0}),
    "split_wide": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 1, moe.MOE_OPT_WIDE_UP: 1}),
    "split_m64": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 0, moe.MOE_OPT_TILE_M: 64}),
    "fused": (moe.MOE_FUSED, {}),
    "fused_dsmem": (moe.MOE_FUSED, {moe.MOE_OPT_FUSED_DSMEM: 1}),
    "fused_splitk": (moe.MOE_FUSED, {moe.MOE_OPT_FUSED_CLUSTER: 0}),
}
DEFAULTS = {moe.MOE_OPT_UP_PAIRS: 0, moe.MOE_OPT_GATHER: 0, moe.MOE_OPT_SWAP_AB: 0, moe.MOE_OPT_FUSED_CLUSTER: 1,
            moe.MOE_OPT_PAIR_MMA: 2, moe.MOE_OPT_PAIR_SWAP: 0, moe.MOE_OPT_WIDE_UP: 0, moe.MOE_OPT_TILE_M: 0,
            moe.MOE_OPT_FUSED_DSMEM: 0, moe.MOE_OPT_HALF_PAIR_M128: 0, moe.MOE_OPT_DOWN_BANDS: 1,
            moe.MOE_OPT_DOWN_EPI8: 1, moe.MOE_OPT_UP_SWAP: 1}
PIPELINES = list(MODES)


def run_mode(inp, dev, mode, **kw):
    pipeline, opts = MODES[mode]
    for o, v in opts.items():
        moe.moe_ffn_set_option(o, v)
    try:
        return run_forward(inp, dev, pipeline=pipeline, **kw)
    finally:
        for o in opts:
            moe.moe_ffn_set_option(o, DEFAULTS[o])


def oracle_out(inp, tokens=None):
    return oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_BF16,
                          tokens=tokens)


@pytest.mark.parametrize("pipeline", PIPELINES)
@pytest.mark.parametrize("T,D,H,E,k,routing", [
    (64, 256, 128, 8, 2, "topk_logits"),      # the tiny workload's shape
    (300, 512, 256, 16, 4, "uniform"),        # ragged tails in every expert
    (1, 256, 128, 4, 4, "uniform"),           # a single token
    (200, 256, 384, 3, 1, "uniform"),         # top-1, H not a multiple of 256
    (129, 768, 256, 40, 8, "zipf"),           # several experts empty
    (512, 2048, 768, 128, 8, "topk_logits"),  # prefill dims, 512 tokens
    (96, 384, 128, 6, 3, "uniform"),          # D % 256 != 0 (split only: 128-column down tiles)
    (200, 256, 128, 1024, 4, "uniform"),      # the largest expert count
    (130, 256, 128, 1, 1, "uniform"),         # one expert, top-1: a dense SwiGLU FFN scaled by w
    (100, 256, 128, 64, 32, "uniform"),       # k = 32 distinct experts per token (fp32 row sums)
    (300, 512, 256, 32, 9, "uniform"),        # the smallest k summed in fp32
    (257, 1024, 256, 64, 16, "zipf"),         # k = 16 with empty experts
])
def test_forward_small(T, D, H, E, k, routing, pipeline):
    if D % 256 and MODES[pipeline][0] != moe.MOE_SPLIT:
        pytest.skip("fused pipeline needs D % 256 == 0")
    inp = wl.make_custom(T, D, H, E, k, seed=T + D, routing=routing)
    out, _ = run_mode(inp, to_dev(inp), pipeline)
    r = assert_close(out, oracle_out(inp), label=f"T={T} D={D} H={H} E={E} k={k}")
    print(f"{pipeline} T={T} D={D} H={H} E={E} k={k}: max_rel={r[0]:.2e} mean_rel={r[1]:.2e} cos={r[2]:.6f}")


@pytest.mark.parametrize("dsmem", [1, 0])          # act in shared memory where the slice fits; the L2 ring
@pytest.mark.parametrize("csize", [1, 2, 4, 8])   # 1: automatic
@pytest.mark.parametrize("T,D,H,E,k", [
    (150, 512, 128, 8, 2),      # 64 or 128 act columns per CTA
    (300, 1024, 512, 16, 4),    # several GEMM1 and GEMM2 sub-chunks per CTA
    (200, 2048, 256, 32, 8),    # 32 act columns per CTA with clusters of 8
    (1000, 2048, 768, 8, 8),    # prefill dims, ~8 row blocks per expert: each ring buffer reused
])
def test_fused_cluster_shapes(T, D, H, E, k, csize, dsmem):
    if csize > 1 and (D % (256 * csize) or (H // csize) % 32):
        pytest.skip("cluster size does not apply to this shape")
    inp = wl.make_custom(T, D, H, E, k, seed=T + H, routing="uniform")
    moe.moe_ffn_set_option(moe.MOE_OPT_FUSED_CLUSTER, csize)
    moe.moe_ffn_set_option(moe.MOE_OPT_FUSED_DSMEM, dsmem)
    try:
        out, _ = run_forward(inp, to_dev(inp), pipeline=moe.MOE_FUSED)
    finally:
        moe.moe_ffn_set_option(moe.MOE_OPT_FUSED_CLUSTER, 1)
        moe.moe_ffn_set_option(moe.MOE_OPT_FUSED_DSMEM, 0)
    r = assert_close(out, oracle_out(inp), label=f"fused C={csize} dsmem={dsmem} T={T} D={D} H={H} E={E} k={k}")
    print(f"fused C={csize} dsmem={dsmem} T={T} D={D} H={H} E={E} k={k}: max_rel={r[0]:.2e} mean_rel={r[1]:.2e} "
          f"cos={r[2]:.6f}")


@pytest.mark.parametrize("pipeline", PIPELINES)
def test_forward_tiny_workload(pipeline):
    inp = wl.make_inputs("tiny", seed=0)
    out, _ = run_mode(inp, to_dev(inp), pipeline)
    assert_close(out, oracle_out(inp), label="tiny")


@pytest.mark.parametrize("pipeline", PIPELINES)
def test_forward_all_tokens_one_expert(pipeline):
    inp = wl.make_custom(600, 256, 256, 8, 2, seed=5, routing="uniform")
    inp["topk_ids"][:, 0] = 3
    inp["topk_ids"][:, 1] = 3          # the same expert twice per token
    out, _ = run_mode(inp, to_dev(inp), pipeline)
    assert_close(out, oracle_out(inp), label="one expert")


@pytest.mark.parametrize("pipeline", PIPELINES)
def test_forward_repeat_calls_and_reused_workspace(pipeline):
    inp = wl.make_custom(100, 256, 128, 8, 2, seed=11)
    dev = to_dev(inp)
    out1, ws = run_mode(inp, dev, pipeline)
    out2, _ = run_mode(inp, dev, pipeline, workspace=ws, out=torch.ones_like(out1))
    ref = oracle_out(inp)
    assert_close(out1, ref, label="first")
    assert_close(out2, ref, label="second (out overwritten, not accumulated)")


def test_zero_tokens_is_a_noop():
    inp = wl.make_custom(4, 256, 128, 4, 2, seed=2)
    dev = to_dev(inp)
    out = torch.zeros(1, 256, dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(4, 4, 256, 128, 2)
    assert moe.moe_ffn_forward(dev["x"], dev["w1"], dev["w2"], dev["topk_ids"], dev["topk_w"], out, E=4, D=256, H=128,
                               k=2, workspace=ws, T=0) == 0
    assert moe.moe_ffn_sync_status(ws) == 0


def test_unsupported_combinations_rejected():
    inp = wl.make_custom(8, 256, 128, 4, 2, seed=1)
    dev = to_dev(inp)
    with pytest.raises(moe.MoeFFNError):  # MXFP8 without scale arrays
        run_forward(inp, dev, pipeline=moe.MOE_SPLIT, dtype=moe.MOE_MXFP8, check_status=False)
    inp = wl.make_custom(8, 384, 128, 4, 2, seed=1)
    with pytest.raises(moe.MoeFFNError):  # fused needs D % 256 == 0
        run_forward(inp, to_dev(inp), pipeline=moe.MOE_FUSED, check_status=False)


@pytest.mark.parametrize("pipeline", PIPELINES)
@pytest.mark.parametrize("name", ["decode", "prefill", "large_skewed"])
def test_forward_full_workload_sampled(name, pipeline):
    """Full-size workloads: decode on every token; prefill and large_skewed on
    the first and last routed token of every expert, the first token of every
    expert's last row block, and 1000 seeded random tokens."""
    if name == "large_skewed" and pipeline not in ("split", "fused", "fused_dsmem", "fused_splitk", "split_pair2",
                                                   "split_wide", "split_m64", "split_pair2_bands"):
        pytest.skip("option variants are covered at the smaller sizes")
    inp = cached_inputs(name)
    out, _ = run_mode(inp, to_dev(inp), pipeline)
    tokens = None if name == "decode" else coverage_tokens(inp["topk_ids"])
    ref = oracle_out(inp, tokens=tokens)
    got = out if tokens is None else out[torch.from_numpy(tokens.astype(np.int64)).cuda()]
    r = assert_close(got, ref, label=name)
    print(f"{pipeline} {name}: {0 if tokens is None else tokens.size} sampled tokens, max_rel={r[0]:.2e} "
          f"mean_rel={r[1]:.2e} cos={r[2]:.6f}")
    assert torch.isfinite(out.float()).all()
