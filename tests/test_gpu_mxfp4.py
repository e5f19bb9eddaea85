"""MXFP4 expert weights ("GC-MoE on SM120" sec. 2.2: E2M1 codes with one
UE8M0 scale per 32 elements) on the MXFP8 path: the device widening of the
codes against e4m3 codes of the format's 16 values (bit-exact), and the
forward pass on widened weights against the oracle's MXFP4 weight mode (act
requantized per 32 along H on both sides) at the MXFP8 tolerances."""
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
