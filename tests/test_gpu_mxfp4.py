"""MXFP4 expert weights ("GC-MoE on SM120" sec. 2.2: E2M1 codes with one
UE8M0 scale per 32 elements) on the MXFP8 path: the device widening of the
codes against e4m3 codes of the format's 16 values (bit-exact), the forward
pass on widened weights, and the forward pass on the packed 4-bit codes
themselves (MOE_MXFP4W: 4-bit tensor maps, E2M1 as the B operand of
kind::mxf8f6f4), each against the oracle's MXFP4 weight mode (act requantized
per 32 along H on both sides) at the MXFP8 tolerances."""
import numpy as np
import pytest
import torch

import grouped_gemm_gb300 as moe
import oracle
from grouped_gemm_gb300 import workloads as wl

from helpers import assert_close
from test_gpu_mxfp8 import run_mx

pytestmark = pytest.mark.gpu

E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def expected_codes(packed):
    """Test-side widening: E2M1 table value of each nibble (low first), cast to
    e4m3 by torch."""
    e4m3 = torch.tensor(E2M1_VALUES, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = e4m3[packed & 0xF]
    out[..., 1::2] = e4m3[packed >> 4]
    return out


def widen(packed):
    src = torch.from_numpy(np.ascontiguousarray(packed)).cuda()
    dst = torch.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=torch.uint8, device="cuda")
    moe.moe_ffn_widen_mxfp4_weights(src, dst)
    torch.cuda.synchronize()
    return dst.cpu().numpy()


def test_widen_bit_exact():
    rng = np.random.default_rng(3)
    every = np.tile(np.arange(256, dtype=np.uint8), 64)                      # each byte value 64 times
    packed = np.concatenate([every, rng.integers(0, 256, 16 * 3001, dtype=np.uint8)])
    assert np.array_equal(widen(packed), expected_codes(packed))


@pytest.mark.parametrize("pipeline", [moe.MOE_SPLIT, moe.MOE_FUSED])
@pytest.mark.parametrize("T,D,H,E,k,routing", [
    (64, 256, 128, 8, 2, "topk_logits"),
    (300, 512, 256, 16, 4, "uniform"),
])
def test_mxfp4_weights_forward(T, D, H, E, k, routing, pipeline):
    inp = wl.make_custom(T, D, H, E, k, seed=T + D, routing=routing, dtype="mxfp4w")
    w1, w2 = widen(inp["w1"]), widen(inp["w2"])
    assert np.array_equal(w1, expected_codes(inp["w1"])) and np.array_equal(w2, expected_codes(inp["w2"]))
    out = run_mx(dict(inp, w1=w1, w2=w2), pipeline)
    ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_MXFP8,
                         x_sf=inp["x_sf"], w1_sf=inp["w1_sf"], w2_sf=inp["w2_sf"], fp4_weights=True)
    r = assert_close(out, ref, dtype="mxfp8", label=f"mxfp4 weights T={T} D={D} H={H}")
    print(f"mxfp4 weights pipeline={pipeline} T={T} D={D} H={H} E={E} k={k}: max_rel={r[0]:.2e} mean_rel={r[1]:.2e}")


def run_mx4(inp, swap=2):
    """moe_ffn_forward with MOE_MXFP4W: the packed codes as they are.  swap:
    MOE_OPT_MX_SWAP (0 the default kernels, 1 the swap-AB ones, 2 automatic)."""
    w = inp["workload"]
    dev = {k: torch.from_numpy(np.ascontiguousarray(inp[k])).cuda() for k in ("x", "x_sf", "w1", "w2")}
    w1p = torch.empty(inp["w1_sf"].size, dtype=torch.uint8, device="cuda")
    w2p = torch.empty(inp["w2_sf"].size, dtype=torch.uint8, device="cuda")
    moe.moe_ffn_prepare_mxfp8_weights(torch.from_numpy(inp["w1_sf"]).cuda(), torch.from_numpy(inp["w2_sf"]).cuda(),
                                      w1p, w2p, w.E, w.D, w.H)
    ids = torch.from_numpy(inp["topk_ids"]).cuda()
    tw = torch.from_numpy(inp["topk_w"]).cuda()
    out = torch.full((w.T, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(w.T, w.E, w.D, w.H, w.k, moe.MOE_MXFP4W, moe.MOE_SPLIT)
    moe.moe_ffn_set_option(moe.MOE_OPT_MX_SWAP, swap)
    try:
        moe.moe_ffn_forward(dev["x"], dev["w1"], dev["w2"], ids, tw, out, E=w.E, D=w.D, H=w.H, k=w.k, workspace=ws,
                            dtype=moe.MOE_MXFP4W, pipeline=moe.MOE_SPLIT, x_sf=dev["x_sf"], w1_sf=w1p, w2_sf=w2p)
    finally:
        moe.moe_ffn_set_option(moe.MOE_OPT_MX_SWAP, 0)
    st = moe.moe_ffn_sync_status(ws)
    assert st == 0, moe.moe_ffn_status_string(st)
    return out


@pytest.mark.parametrize("swap", [0, 1])       # the swap-AB kernels (weights on the M side), or not
@pytest.mark.parametrize("T,D,H,E,k,routing", [
    (64, 256, 128, 8, 2, "topk_logits"),
    (300, 512, 256, 16, 4, "uniform"),
    (1, 256, 384, 4, 4, "uniform"),
    (129, 768, 256, 40, 8, "zipf"),          # several experts empty
    (100, 256, 256, 64, 32, "uniform"),      # k = 32: rows of a token summed in fp32 (never swapped)
    (700, 512, 256, 4, 2, "uniform"),        # ~350 rows per expert: full 128-row blocks and a ragged one
])
def test_mxfp4_packed_weights_forward(T, D, H, E, k, routing, swap):
    inp = wl.make_custom(T, D, H, E, k, seed=T + H, routing=routing, dtype="mxfp4w")
    out = run_mx4(inp, swap)
    ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_MXFP8,
                         x_sf=inp["x_sf"], w1_sf=inp["w1_sf"], w2_sf=inp["w2_sf"], fp4_weights=True)
    r = assert_close(out, ref, dtype="mxfp8", label=f"packed mxfp4 weights swap={swap} T={T} D={D} H={H} E={E} k={k}")
    print(f"packed mxfp4 swap={swap} T={T} D={D} H={H} E={E} k={k}: max_rel={r[0]:.2e} mean_rel={r[1]:.2e} "
          f"cos={r[2]:.6f}")


@pytest.mark.parametrize("swap", [0, 2])       # the default kernels; automatic (the swap-AB ones here)
def test_mxfp4_packed_weights_decode_workload(swap):
    """The decode workload's shape (T=64, D=6144, H=2048, E=32, k=8) with MXFP4
    weights, every token checked: the weight stream that 4-bit codes halve."""
    inp = wl.make_inputs("decode_mxfp4w", seed=0)
    out = run_mx4(inp, swap)
    ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_MXFP8,
                         x_sf=inp["x_sf"], w1_sf=inp["w1_sf"], w2_sf=inp["w2_sf"], fp4_weights=True)
    r = assert_close(out, ref, dtype="mxfp8", label="packed mxfp4 weights, decode workload")
    print(f"packed mxfp4 decode: max_rel={r[0]:.2e} mean_rel={r[1]:.2e} cos={r[2]:.6f}")
