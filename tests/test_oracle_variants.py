"""Pins for the oracle's activation and shared-expert variants (CPU only).

Clamped SwiGLU ("Porting Block-Scaled GEMM Kernels from Blackwell to Rubin"
sec. 5.3: an upper bound on the gate, a two-sided bound on the up projection,
then silu(gate) * up): the one-expert, weight-1 case is the dense clamped FFN
written with torch's clamp and silu in fp64; a limit above every |gate| and
|up| leaves the plain SwiGLU; the clamp bounds |act| by 0.2785 * limit for a
small limit.  Shared experts (GC-MoE on SM120 sec. 4.7: a shared expert runs
on every token): an expert that every token uses with weight 1 adds exactly
the dense FFN of that expert to the routed output."""
import numpy as np
import pytest
import torch

import oracle
from grouped_gemm_gb300 import workloads as wl

from test_oracle_pins import bf16_bits_to_f64, dense_ffn_torch, rel_err


def dense_clamped_torch(x, w1, w2, H, limit):
    g = torch.clamp(x @ w1[:H].T, max=limit)
    u = torch.clamp(x @ w1[H:].T, min=-limit, max=limit)
    return (torch.nn.functional.silu(g) * u) @ w2.T


@pytest.mark.parametrize("limit", [0.05, 0.2, 0.5])
def test_clamped_top1_is_dense_clamped_ffn(limit):
    inp = wl.make_custom(T=40, D=64, H=32, E=1, k=1, seed=12)
    # make gate / up large enough that the clamp is active for a fraction of them
    x = torch.from_numpy(bf16_bits_to_f64(inp["x"]))
    w1 = torch.from_numpy(bf16_bits_to_f64(inp["w1"][0]))
    w2 = torch.from_numpy(bf16_bits_to_f64(inp["w2"][0]))
    g = x @ w1[:32].T
    assert (g > limit).any() and (g < limit).any()
    ours = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], np.ones((40, 1), np.float32),
                          act=oracle.ACT_EXACT, swiglu_limit=limit)
    ref = dense_clamped_torch(x, w1, w2, 32, limit).numpy()
    assert rel_err(ours, ref) < 1e-12


def test_clamp_above_every_value_is_plain_swiglu():
    inp = wl.make_custom(T=30, D=128, H=64, E=4, k=2, seed=13)
    plain = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_BF16)
    big = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_BF16,
                         swiglu_limit=1e30)
    assert np.array_equal(plain, big)


def test_small_clamp_bounds_the_activation():
    # |silu(g) * u| <= max_{g <= L} |g sigmoid(g)| * L <= 0.2785 L for small L, so the
    # output is bounded by 0.2785 L * sum_h |W2[e][d][h]| * sum_j |w_j|
    inp = wl.make_custom(T=20, D=64, H=32, E=3, k=2, seed=14)
    L = 1e-3
    out = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_EXACT,
                         swiglu_limit=L)
    w2 = bf16_bits_to_f64(inp["w2"])
    bound = 0.2785 * L * np.abs(w2).sum(axis=2).max() * np.abs(inp["topk_w"]).sum(axis=1).max()
    assert np.abs(out).max() <= bound
    assert np.abs(out).max() > 0.05 * bound


def test_shared_expert_adds_its_dense_ffn():
    T, D, H, E, k = 33, 64, 32, 5, 2
    inp = wl.make_custom(T=T, D=D, H=H, E=E + 1, k=k, seed=15, routing="uniform")
    ids = inp["topk_ids"] % E                       # routed experts 0..E-1
    routed = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], ids, inp["topk_w"], act=oracle.ACT_EXACT)
    ids_ext = np.concatenate([ids, np.full((T, 1), E, np.int32)], axis=1)
    w_ext = np.concatenate([inp["topk_w"], np.ones((T, 1), np.float32)], axis=1)
    both = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], ids_ext, w_ext, act=oracle.ACT_EXACT)
    x = torch.from_numpy(bf16_bits_to_f64(inp["x"]))
    shared = dense_ffn_torch(x, torch.from_numpy(bf16_bits_to_f64(inp["w1"][E])),
                             torch.from_numpy(bf16_bits_to_f64(inp["w2"][E])), H).numpy()
    assert rel_err(both, routed + shared) < 1e-12
