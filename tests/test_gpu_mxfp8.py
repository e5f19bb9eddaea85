"""MXFP8 path ("Prime Flash MoE" sec. 7): the device requantizer against the
oracle's codec (bit-exact: both decide in fp32), the weight-scale repacking
against its documented tile layout, and the forward pass against the fp64
oracle (act requantized per 32 along H on both sides) at the parity
MXFP8 tolerances (max 4e-2, mean 1e-2)."""
import numpy as np
import pytest
import torch

import grouped_gemm_gb300 as moe
import oracle
from grouped_gemm_gb300 import workloads as wl

from helpers import assert_close, cached_inputs, coverage_tokens

pytestmark = pytest.mark.gpu


def edge_values(rng):
    blocks = []
    for p in range(-30, 30, 3):
        for m in (1.0, 1.75, np.nextafter(np.float32(1.75), np.float32(2)), 1.5, np.nextafter(np.float32(2), 0)):
            b = rng.standard_normal(32) * (2.0 ** p)
            b[rng.integers(0, 32)] = m * 2.0 ** p * (1 if rng.random() < 0.5 else -1)
            blocks.append(b)
    blocks.append(np.zeros(32))
    one = np.zeros(32)
    one[5] = 3.0
    blocks.append(one)
    # values that land exactly between two e4m3 codes after scaling
    codes = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = ((codes[:-1] + codes[1:]) / 2)[:-1]
    for i in range(0, len(mids) - 31, 31):
        b = mids[i:i + 32].copy()
        b[0] = 448.0        # fixes the block scale at 2^0
        blocks.append(b)
    blocks.append(rng.standard_normal(32 * 64).reshape(-1, 32) * 0.01)
    return np.concatenate([np.atleast_2d(b) for b in blocks]).astype(np.float32).ravel()


def test_device_requantizer_matches_oracle_bit_exact():
    rng = np.random.default_rng(0)
    v = edge_values(rng)
    v = np.concatenate([v, rng.standard_normal(32 * 4096).astype(np.float32) * np.float32(3)])
    x = torch.from_numpy(v).cuda()
    q = torch.empty(v.size, dtype=torch.uint8, device="cuda")
    sf = torch.empty(v.size // 32, dtype=torch.uint8, device="cuda")
    moe.moe_ffn_debug_mx_quantize(x, q, sf)
    torch.cuda.synchronize()
    rq, rsf, _ = oracle.mx_quantize(v.astype(np.float64))
    assert np.array_equal(sf.cpu().numpy(), rsf)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_weight_scale_repacking_layout():
    E, D, H = 2, 256, 384
    rng = np.random.default_rng(1)
    w1_sf = rng.integers(100, 140, size=(E, 2 * H, D // 32), dtype=np.uint8)
    w2_sf = rng.integers(100, 140, size=(E, D, H // 32), dtype=np.uint8)
    p1 = torch.zeros(w1_sf.size, dtype=torch.uint8, device="cuda")
    p2 = torch.zeros(w2_sf.size, dtype=torch.uint8, device="cuda")
    moe.moe_ffn_prepare_mxfp8_weights(torch.from_numpy(w1_sf).cuda(), torch.from_numpy(w2_sf).cuda(), p1, p2, E, D, H)
    torch.cuda.synchronize()

    def expected(sf):  # 512-byte tiles of 128 rows x 4 scales, row r at (r%32)*16 + (r//32)*4
        rows, k32 = sf.reshape(-1, sf.shape[-1]).shape
        out = np.zeros(rows * k32, np.uint8)
        flat = sf.reshape(rows, k32)
        for r in range(rows):
            for c in range(k32):
                kt, g = divmod(c, 4)
                tile = (r // 128) * (k32 // 4) + kt
                out[tile * 512 + (r % 128 % 32) * 16 + (r % 128 // 32) * 4 + g] = flat[r, c]
        return out

    assert np.array_equal(p1.cpu().numpy(), expected(w1_sf))
    assert np.array_equal(p2.cpu().numpy(), expected(w2_sf))


def run_mx(inp, pipeline=moe.MOE_SPLIT, cluster=1, bands=1, pairs=0, swap=0, check=True):
    """cluster: MOE_OPT_FUSED_CLUSTER for the call (1 automatic, 2/4/8 that
    size, 0 the fused kernel with fp32 partial sums); bands:
    MOE_OPT_DOWN_BANDS (token-band order of the split down kernel's tiles);
    pairs: MOE_OPT_MX_PAIRS (split GEMMs on CTA pairs: 0 off, 1 on, 2 automatic);
    swap: MOE_OPT_MX_SWAP (swap-AB split GEMMs: 0 off, 1 on, 2 automatic).
    check=False returns (out, status) instead of asserting a clean status."""
    w = inp["workload"]
    dev = {k: torch.from_numpy(inp[k]).cuda() for k in ("x", "x_sf", "w1", "w2")}
    w1p = torch.empty(inp["w1_sf"].size, dtype=torch.uint8, device="cuda")
    w2p = torch.empty(inp["w2_sf"].size, dtype=torch.uint8, device="cuda")
    moe.moe_ffn_prepare_mxfp8_weights(torch.from_numpy(inp["w1_sf"]).cuda(), torch.from_numpy(inp["w2_sf"]).cuda(),
                                      w1p, w2p, w.E, w.D, w.H)
    ids = torch.from_numpy(inp["topk_ids"]).cuda()
    tw = torch.from_numpy(inp["topk_w"]).cuda()
    out = torch.full((w.T, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(w.T, w.E, w.D, w.H, w.k, moe.MOE_MXFP8, pipeline)
    moe.moe_ffn_set_option(moe.MOE_OPT_FUSED_CLUSTER, cluster)
    moe.moe_ffn_set_option(moe.MOE_OPT_DOWN_BANDS, bands)
    moe.moe_ffn_set_option(moe.MOE_OPT_MX_PAIRS, pairs)
    moe.moe_ffn_set_option(moe.MOE_OPT_MX_SWAP, swap)
    try:
        moe.moe_ffn_forward(dev["x"], dev["w1"], dev["w2"], ids, tw, out, E=w.E, D=w.D, H=w.H, k=w.k, workspace=ws,
                            dtype=moe.MOE_MXFP8, pipeline=pipeline, x_sf=dev["x_sf"], w1_sf=w1p, w2_sf=w2p)
    finally:
        moe.moe_ffn_set_option(moe.MOE_OPT_FUSED_CLUSTER, 1)
        moe.moe_ffn_set_option(moe.MOE_OPT_DOWN_BANDS, 1)
        moe.moe_ffn_set_option(moe.MOE_OPT_MX_PAIRS, 0)
        moe.moe_ffn_set_option(moe.MOE_OPT_MX_SWAP, 0)
    st = moe.moe_ffn_sync_status(ws)
    if not check:
        return out, st
    assert st == 0, moe.moe_ffn_status_string(st)
    return out


def oracle_mx(inp, tokens=None):
    return oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_MXFP8,
                          x_sf=inp["x_sf"], w1_sf=inp["w1_sf"], w2_sf=inp["w2_sf"], tokens=tokens)


# split: the default (single-CTA kernels); split_swap: the swap-AB kernels;
# split_swap_auto: the automatic swap choice (swap-AB where an expert holds at
# most 64 rows on average);
# split_pairs: the CTA-pair kernels;
# split_auto: pairs chosen automatically (single CTAs at the small shapes, pairs
# at full size); fused: on clusters
# (automatic size); fused_splitk: H split over CTAs with fp32 partial sums;
# split_bands: the down kernel's tiles in the order of three token bands
PIPES = {"split": (moe.MOE_SPLIT, 1), "split_swap": (moe.MOE_SPLIT, 1, 1, 0, 1),
         "split_swap_auto": (moe.MOE_SPLIT, 1, 1, 0, 2), "split_pairs": (moe.MOE_SPLIT, 1, 1, 1),
         "split_auto": (moe.MOE_SPLIT, 1, 1, 2), "fused": (moe.MOE_FUSED, 1), "fused_splitk": (moe.MOE_FUSED, 0),
         "split_bands": (moe.MOE_SPLIT, 1, 3), "split_pairs_bands": (moe.MOE_SPLIT, 1, 3, 1)}


@pytest.mark.parametrize("pipe", list(PIPES))
@pytest.mark.parametrize("T,D,H,E,k,routing", [
    (64, 256, 128, 8, 2, "topk_logits"),
    (300, 512, 256, 16, 4, "uniform"),
    (1, 256, 384, 4, 4, "uniform"),
    (129, 768, 256, 40, 8, "zipf"),
    (512, 1024, 512, 16, 8, "uniform"),
    (100, 256, 256, 64, 32, "uniform"),     # k = 32: rows of a token summed in fp32
    (300, 512, 256, 32, 12, "zipf"),        # k = 12 with empty experts
])
def test_mxfp8_forward_small(T, D, H, E, k, routing, pipe):
    inp = wl.make_custom(T, D, H, E, k, seed=T + H, routing=routing, dtype="mxfp8")
    out = run_mx(inp, *PIPES[pipe])
    r = assert_close(out, oracle_mx(inp), dtype="mxfp8", label=f"mxfp8 {pipe} T={T} D={D} H={H}")
    print(f"mxfp8 {pipe} T={T} D={D} H={H} E={E} k={k}: max_rel={r[0]:.2e} mean_rel={r[1]:.2e} cos={r[2]:.6f}")


@pytest.mark.parametrize("pipe", list(PIPES))
def test_mxfp8_full_workload_sampled(pipe):
    # every expert's first, last and tail-block rows plus 1000 seeded random tokens
    if pipe in ("split_auto", "split_swap", "split_swap_auto"):
        pytest.skip("at full size: the CTA pairs (split_pairs) or the single-CTA kernels (split)")
    inp = cached_inputs("mxfp8")
    out = run_mx(inp, *PIPES[pipe])
    tokens = coverage_tokens(inp["topk_ids"], seed=2)
    r = assert_close(out[torch.from_numpy(tokens.astype(np.int64)).cuda()], oracle_mx(inp, tokens), dtype="mxfp8",
                     label="mxfp8 workload")
    print(f"mxfp8 workload {pipe}: {tokens.size} tokens, max_rel={r[0]:.2e} mean_rel={r[1]:.2e} cos={r[2]:.6f}")
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("csize", [2, 4, 8])
@pytest.mark.parametrize("T,D,H,E,k", [
    (512, 1024, 512, 16, 8),     # several GEMM1 and GEMM2 sub-chunks per CTA
    (1000, 2048, 1024, 8, 8),    # ~8 row blocks per expert: each ring buffer reused
])
def test_mxfp8_fused_cluster_sizes(T, D, H, E, k, csize):
    if D % (256 * csize) or H % (128 * csize):
        pytest.skip("cluster size does not apply to this shape")
    inp = wl.make_custom(T, D, H, E, k, seed=T + D, routing="uniform", dtype="mxfp8")
    out = run_mx(inp, moe.MOE_FUSED, cluster=csize)
    r = assert_close(out, oracle_mx(inp), dtype="mxfp8", label=f"mxfp8 fused C={csize} T={T} D={D} H={H}")
    print(f"mxfp8 fused C={csize} T={T} D={D} H={H} E={E} k={k}: max_rel={r[0]:.2e} mean_rel={r[1]:.2e}")


@pytest.mark.parametrize("pairs,swap", [(0, 0), (1, 0), (0, 1)])
def test_mxfp8_wait_timeout_is_reported_and_context_survives(pairs, swap):
    # the MMA issuer of the single-CTA (pairs 0) or CTA-pair (pairs 1) MXFP8
    # kernels first waits on a barrier nothing arrives on (MOE_OPT_TEST_STALL
    # 1); with a 1 ms bound the wait runs out, the status reads
    # MOE_ERR_DEVICE_TIMEOUT, and the next call is correct
    inp = wl.make_custom(300, 512, 256, 16, 4, seed=3, routing="uniform", dtype="mxfp8")
    moe.moe_ffn_set_wait_limit_ns(1_000_000)
    moe.moe_ffn_set_option(moe.MOE_OPT_TEST_STALL, 1)
    try:
        _, st = run_mx(inp, pairs=pairs, swap=swap, check=False)
    finally:
        moe.moe_ffn_set_option(moe.MOE_OPT_TEST_STALL, 0)
        moe.moe_ffn_set_wait_limit_ns(2_000_000_000)
    assert st == 6, moe.moe_ffn_status_string(st)
    out = run_mx(inp, pairs=pairs, swap=swap)
    assert_close(out, oracle_mx(inp), dtype="mxfp8", label=f"mxfp8 after timeout pairs={pairs} swap={swap}")
