"""NVFP4 forward pass (moe_ffn_forward_nvfp4: E2M1 codes with one E4M3 scale
per 16 elements and fp32 global scales, "Porting Block-Scaled GEMM Kernels from
Blackwell to Rubin" sec. 1.2, 6.1; GEMMs on kind::mxf4nvf4.block_scale
.scale_vec::4X) against the oracle's NVFP4 mode with act requantized to NVFP4
by the same rule and global scale on both sides.

Tolerance: the bf16 parity bounds (max 2e-2, mean 5e-3).  No bound is stated
for NVFP4; the GPU and the oracle quantize from the same decoded
operands, so they differ only by fp32 against fp64 accumulation, the rare act
code that the two precisions round to opposite sides of a decision boundary,
and the bf16 output and its reductions -- the bf16 bounds' own sources."""
import numpy as np
import pytest
import torch

import grouped_gemm_gb300 as moe
import oracle
from grouped_gemm_gb300 import workloads as wl

from helpers import assert_close

pytestmark = pytest.mark.gpu

ACT_GS = 4.0 / (6 * 448)   # act blocks of amax up to 4 keep their scale below the e4m3 maximum


def run_nv(inp, act_gs=ACT_GS):
    w = inp["workload"]
    T, D, H, E, k = w.T, w.D, w.H, w.E, w.k
    dev = {key: torch.from_numpy(np.ascontiguousarray(inp[key])).cuda() for key in ("x", "x_sf", "w1", "w2")}
    w1p = torch.empty(inp["w1_sf"].size, dtype=torch.uint8, device="cuda")
    w2p = torch.empty(inp["w2_sf"].size, dtype=torch.uint8, device="cuda")
    moe.moe_ffn_prepare_nvfp4_weights(torch.from_numpy(inp["w1_sf"]).cuda(), torch.from_numpy(inp["w2_sf"]).cuda(),
                                      w1p, w2p, E, D, H)
    gs = {"x_gs": torch.tensor([float(inp["x_gs"])], dtype=torch.float32, device="cuda"),
          "w1_gs": torch.from_numpy(inp["w1_gs"]).cuda(), "w2_gs": torch.from_numpy(inp["w2_gs"]).cuda(),
          "act_gs": torch.tensor([act_gs], dtype=torch.float32, device="cuda")}
    ids = torch.from_numpy(inp["topk_ids"]).cuda()
    tw = torch.from_numpy(inp["topk_w"]).cuda()
    out = torch.full((T, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(T, E, D, H, k, moe.MOE_NVFP4, moe.MOE_SPLIT)
    moe.moe_ffn_forward_nvfp4(dev["x"], dev["x_sf"], dev["w1"], w1p, dev["w2"], w2p, gs["x_gs"], gs["w1_gs"],
                              gs["w2_gs"], gs["act_gs"], ids, tw, out, E=E, D=D, H=H, k=k, workspace=ws)
    st = moe.moe_ffn_sync_status(ws)
    assert st == 0, moe.moe_ffn_status_string(st)
    return out


def oracle_nv(inp, act_gs=ACT_GS, tokens=None):
    return oracle.moe_ffn_nvfp4(inp["x"], inp["x_sf"], float(inp["x_gs"]), inp["w1"], inp["w1_sf"], inp["w1_gs"],
                                inp["w2"], inp["w2_sf"], inp["w2_gs"], inp["topk_ids"], inp["topk_w"],
                                act=oracle.ACT_NVFP4, act_gs=act_gs, tokens=tokens)


@pytest.mark.parametrize("T,D,H,E,k,routing", [
    (64, 256, 256, 8, 2, "topk_logits"),
    (300, 512, 512, 16, 4, "uniform"),
    (1, 256, 256, 4, 4, "uniform"),          # a single token
    (129, 768, 256, 40, 8, "zipf"),          # several experts empty
    (100, 256, 256, 64, 32, "uniform"),      # k = 32: rows of a token summed in fp32
    (512, 2048, 768, 32, 8, "uniform"),      # prefill dims, several row blocks per expert
])
def test_nvfp4_forward(T, D, H, E, k, routing):
    inp = wl.make_custom(T, D, H, E, k, seed=T + H, routing=routing, dtype="nvfp4")
    out = run_nv(inp)
    r = assert_close(out, oracle_nv(inp), dtype="bf16", label=f"nvfp4 T={T} D={D} H={H} E={E} k={k}")
    print(f"nvfp4 T={T} D={D} H={H} E={E} k={k}: max_rel={r[0]:.2e} mean_rel={r[1]:.2e} cos={r[2]:.6f}")


def test_nvfp4_global_scales_enter_both_epilogues():
    # doubling every weight global scale doubles gate and up (and so changes
    # act nonlinearly) and doubles W2's contribution; the result must follow
    # the oracle with the same scales, and differ from the unscaled one
    inp = wl.make_custom(96, 512, 256, 8, 2, seed=7, dtype="nvfp4")
    base = run_nv(inp).float().cpu().numpy()
    inp2 = dict(inp, w1_gs=(inp["w1_gs"] * 2).astype(np.float32), w2_gs=(inp["w2_gs"] * 2).astype(np.float32))
    out2 = run_nv(inp2)
    assert_close(out2, oracle_nv(inp2), dtype="bf16", label="doubled global scales")
    assert np.abs(out2.float().cpu().numpy() - base).sum() > 0.5 * np.abs(base).sum()


def test_nvfp4_rejects_bad_shapes():
    inp = wl.make_custom(8, 256, 256, 4, 2, seed=1, dtype="nvfp4")
    with pytest.raises(moe.MoeFFNError):   # H % 256 != 0
        bad = wl.make_custom(8, 256, 384, 4, 2, seed=1, dtype="nvfp4")
        run_nv(bad)
    assert moe.moe_ffn_workspace_size(8, 4, 256, 256, 2, moe.MOE_NVFP4, moe.MOE_FUSED) == 0
    assert run_nv(inp) is not None


def test_nvfp4_decode_workload():
    """The decode shape (T=64, D=6144, H=2048, E=32, k=8) with NVFP4 operands,
    every token checked, act's global scale the workload's."""
    inp = wl.make_inputs("decode_nvfp4", seed=0)
    act_gs = float(inp["act_gs"])
    out = run_nv(inp, act_gs=act_gs)
    r = assert_close(out, oracle_nv(inp, act_gs=act_gs), dtype="bf16", label="nvfp4 decode workload")
    print(f"nvfp4 decode: max_rel={r[0]:.2e} mean_rel={r[1]:.2e} cos={r[2]:.6f}")
