"""The router step on the GPU (moe_ffn_router_topk, and moe_ffn_forward_logits
which fuses it into the routing launch) against the CPU oracle's router.

Selected expert ids are integer decisions taken on the same fp32 logits on
both sides, so they must match bit for bit.  Weights: the kernel computes the
softmax of the selected logits in fp32 (expf within 2 ulp, a sum of at most
1024 terms in at most 42 roundings, one division), so each weight is within
about 3e-6 relative of the fp64 oracle; the test allows 1e-5 relative.
Forward outputs use the bf16 parity tolerances against the oracle's
forward pass on the oracle's own ids and weights."""
import numpy as np
import pytest
import torch

import grouped_gemm_gb300 as moe
import oracle
from grouped_gemm_gb300 import workloads as wl

from helpers import assert_close, cached_inputs, coverage_tokens, to_dev

pytestmark = pytest.mark.gpu

W_RTOL = 1e-5


def gpu_router(lg, k):
    T, E = lg.shape
    d = torch.from_numpy(lg).cuda()
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_ffn_router_topk(d, k, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


def check(lg, k, gids, gw):
    rids, rw = oracle.router_topk(lg, k)
    assert np.array_equal(gids, rids), np.argwhere(gids != rids)[:5]
    np.testing.assert_allclose(gw.astype(np.float64), rw, rtol=W_RTOL, atol=0)


@pytest.mark.parametrize("T,E,k", [
    (1, 8, 2), (77, 8, 8), (500, 32, 4), (300, 60, 7), (4096, 128, 8), (257, 256, 33),
    (100, 1000, 8), (64, 1024, 1024), (129, 33, 33), (1000, 512, 64),
])
def test_router_matches_oracle(T, E, k):
    lg = wl.router_logits(T, E, seed=T + E + k)
    check(lg, k, *gpu_router(lg, k))


def test_router_ties_nan_and_infinities():
    rng = np.random.default_rng(5)
    lg = rng.integers(-2, 3, size=(200, 96)).astype(np.float32)   # many exact ties
    lg[3, :] = -np.inf
    lg[4, :] = np.nan
    lg[5, ::2] = np.nan
    lg[6, 10] = np.inf
    lg[7, :50] = -np.inf
    for k in (1, 5, 32, 96):
        check(lg, k, *gpu_router(lg, k))


def test_router_rejects_bad_k():
    lg = torch.zeros(4, 8, device="cuda")
    ids = torch.empty(4, 9, dtype=torch.int32, device="cuda")
    w = torch.empty(4, 9, device="cuda")
    with pytest.raises(moe.MoeFFNError):
        moe.moe_ffn_router_topk(lg, 9, ids, w)


PIPES = {"split": moe.MOE_SPLIT, "fused": moe.MOE_FUSED}


@pytest.mark.parametrize("fused_router", [0, 1])  # router launch of its own / inside single-block routing
@pytest.mark.parametrize("pipe", list(PIPES))
@pytest.mark.parametrize("T,D,H,E,k", [
    (64, 256, 128, 8, 2),       # the tiny workload's shape: single-block routing
    (700, 512, 256, 16, 4),     # several routing blocks
    (2048, 2048, 768, 128, 8),  # prefill dims: multi-block routing, every expert live
    (150, 256, 128, 300, 2),    # E > 256: multi-block routing, most experts empty
])
def test_forward_from_logits(T, D, H, E, k, pipe, fused_router):
    moe.moe_ffn_set_option(moe.MOE_OPT_ROUTER_FUSED, fused_router)
    try:
        _forward_from_logits(T, D, H, E, k, pipe)
    finally:
        moe.moe_ffn_set_option(moe.MOE_OPT_ROUTER_FUSED, 0)


def _forward_from_logits(T, D, H, E, k, pipe):
    inp = wl.make_custom(T, D, H, E, k, seed=T + E, routing="uniform")
    lg = wl.router_logits(T, E, seed=T * 3 + k)
    rids, rw = oracle.router_topk(lg, k)
    dev = to_dev(inp)
    ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    out = torch.full((T, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(T, E, D, H, k, moe.MOE_BF16, PIPES[pipe])
    for _ in range(2):  # a second call on the same workspace gives the same result
        moe.moe_ffn_forward_logits(dev["x"], dev["w1"], dev["w2"], torch.from_numpy(lg).cuda(), ids, w, out, E=E,
                                   D=D, H=H, k=k, workspace=ws, pipeline=PIPES[pipe])
        assert moe.moe_ffn_sync_status(ws) == 0
        assert np.array_equal(ids.cpu().numpy(), rids)
        np.testing.assert_allclose(w.cpu().numpy().astype(np.float64), rw, rtol=W_RTOL, atol=0)
        ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], rids, rw.astype(np.float32), act=oracle.ACT_BF16)
        assert_close(out, ref, label=f"from logits {pipe} T={T} E={E} k={k}")


def test_forward_from_logits_mxfp8():
    inp = wl.make_custom(300, 512, 256, 16, 4, seed=3, dtype="mxfp8", routing="uniform")
    T, D, H, E, k = 300, 512, 256, 16, 4
    lg = wl.router_logits(T, E, seed=17)
    rids, rw = oracle.router_topk(lg, k)
    dev = to_dev(inp)
    w1p = torch.empty(inp["w1_sf"].size, dtype=torch.uint8, device="cuda")
    w2p = torch.empty(inp["w2_sf"].size, dtype=torch.uint8, device="cuda")
    moe.moe_ffn_prepare_mxfp8_weights(dev["w1_sf"], dev["w2_sf"], w1p, w2p, E, D, H)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    for pipe in (moe.MOE_SPLIT, moe.MOE_FUSED):
        out = torch.full((T, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        ws = moe.alloc_workspace(T, E, D, H, k, moe.MOE_MXFP8, pipe)
        moe.moe_ffn_forward_logits(dev["x"], dev["w1"], dev["w2"], torch.from_numpy(lg).cuda(), ids, w, out, E=E,
                                   D=D, H=H, k=k, workspace=ws, dtype=moe.MOE_MXFP8, pipeline=pipe,
                                   x_sf=dev["x_sf"], w1_sf=w1p, w2_sf=w2p)
        assert moe.moe_ffn_sync_status(ws) == 0
        assert np.array_equal(ids.cpu().numpy(), rids)
        ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], rids, rw.astype(np.float32), act=oracle.ACT_MXFP8,
                             x_sf=inp["x_sf"], w1_sf=inp["w1_sf"], w2_sf=inp["w2_sf"])
        assert_close(out, ref, dtype="mxfp8", label=f"mxfp8 from logits pipeline={pipe}")


@pytest.mark.parametrize("pipe", list(PIPES))
def test_forward_from_logits_full_prefill(pipe):
    """The prefill workload (T=4096, D=2048, H=768, E=128, k=8) started from
    router logits: ids bit-exact and weights within W_RTOL of the oracle's
    router; the output on every expert's first, last and tail-block rows plus
    1000 seeded random tokens."""
    inp = cached_inputs("prefill")
    w = inp["workload"]
    T, D, H, E, k = w.T, w.D, w.H, w.E, w.k
    lg = wl.router_logits(T, E, seed=1000)
    rids, rw = oracle.router_topk(lg, k)
    dev = to_dev(inp)
    ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    tw = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    out = torch.full((T, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(T, E, D, H, k, moe.MOE_BF16, PIPES[pipe])
    moe.moe_ffn_forward_logits(dev["x"], dev["w1"], dev["w2"], torch.from_numpy(lg).cuda(), ids, tw, out, E=E, D=D,
                               H=H, k=k, workspace=ws, pipeline=PIPES[pipe])
    assert moe.moe_ffn_sync_status(ws) == 0
    assert np.array_equal(ids.cpu().numpy(), rids)
    np.testing.assert_allclose(tw.cpu().numpy().astype(np.float64), rw, rtol=W_RTOL, atol=0)
    tokens = coverage_tokens(rids, seed=3)
    ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], rids, tw.cpu().numpy(), act=oracle.ACT_BF16, tokens=tokens)
    assert_close(out[torch.from_numpy(tokens.astype(np.int64)).cuda()], ref, label=f"prefill from logits {pipe}")
    assert torch.isfinite(out.float()).all()
