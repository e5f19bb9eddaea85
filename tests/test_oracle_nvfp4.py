"""Pins for the oracle's NVFP4 mode: E2M1 codes with one E4M3 scale per 16
elements and a global fp32 scale per tensor (per expert for the weights):
"Porting Block-Scaled GEMM Kernels from Blackwell to Rubin" sec. 1.2 (16
scales per 256-element row) and sec. 5.3 (gate and up dequantized by the
expert's global scale alpha).  Each test checks the oracle against something
other than itself: the input generator's independent numpy encoder, a dense
fp64 SwiGLU FFN on values decoded here from the E2M1 table and torch's e4m3
decode, exact scaling identities, and bit-identity with the MXFP8 mode on
values both formats hold.  CPU only."""
import numpy as np
import torch

import oracle
from grouped_gemm_gb300 import workloads as wl

E2M1_TABLE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                       -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def unpack(packed):
    v = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,))
    v[..., 0::2] = E2M1_TABLE[packed & 0xF]
    v[..., 1::2] = E2M1_TABLE[packed >> 4]
    return v


def e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


def decode_nv4(packed, sf, gs):
    """Test-side decode: table value x e4m3 block scale (per 16) x global scale."""
    return unpack(packed) * np.repeat(e4m3(sf), 16, axis=-1) * np.asarray(gs, np.float64)


def rel_err(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


def dense_swiglu(x, w1, w2, H):
    g = x @ w1[:H].T
    u = x @ w1[H:].T
    return (g / (1.0 + np.exp(-g)) * u) @ w2.T


def run(inp, **kw):
    return oracle.moe_ffn_nvfp4(inp["x"], inp["x_sf"], inp["x_gs"], inp["w1"], inp["w1_sf"], inp["w1_gs"], inp["w2"],
                                inp["w2_sf"], inp["w2_gs"], inp["topk_ids"], inp["topk_w"], **kw)


def test_quantizer_agrees_with_generator_encoder():
    rng = np.random.default_rng(50)
    a = (rng.standard_normal((48, 256)) * 10.0 ** rng.integers(-2, 3, (48, 1))).astype(np.float32)
    for gs in (wl.nv4_global_scale(a), np.float32(1.0), np.float32(0.01)):
        packed, sf = wl.nv4_encode_rows(a, gs)
        q, osf, deq = oracle.nv4_quantize(a.astype(np.float64), float(gs))
        assert np.array_equal(osf, sf.ravel())
        assert np.array_equal(q, packed.ravel())
        assert np.array_equal(deq, decode_nv4(packed, sf, gs).ravel())


def test_quantizer_edge_blocks():
    # all-zero block: scale code 0, codes 0
    q, sf, deq = oracle.nv4_quantize(np.zeros(16), 1.0)
    assert not q.any() and sf[0] == 0 and not deq.any()
    # a block beyond the range: the scale saturates at 448 and the codes at 6
    q, sf, deq = oracle.nv4_quantize(np.full(16, 1e6), 1.0)
    assert sf[0] == 0x7E and deq[0] == 6.0 * 448.0
    # the largest element of a block lands on the top of the E2M1 range when
    # amax / 6 is an e4m3 value
    v = np.linspace(-1.0, 1.0, 16) * 3.0        # amax 3 -> scale 0.5 exactly
    q, sf, deq = oracle.nv4_quantize(v, 1.0)
    assert e4m3(sf)[0] == 0.5 and deq[0] == -3.0 and deq[-1] == 3.0


def test_dense_single_expert():
    """top-1 with weight 1 over one expert is that expert's dense SwiGLU FFN
    on the decoded operands (exact act)."""
    T, D, H = 7, 64, 96
    inp = wl.make_custom(T=T, D=D, H=H, E=1, k=1, seed=51, routing="uniform", dtype="nvfp4")
    inp["topk_w"] = np.ones((T, 1), np.float32)
    got = run(inp, act=oracle.ACT_EXACT)
    x = decode_nv4(inp["x"], inp["x_sf"], inp["x_gs"])
    w1 = decode_nv4(inp["w1"][0], inp["w1_sf"][0], inp["w1_gs"][0])
    w2 = decode_nv4(inp["w2"][0], inp["w2_sf"][0], inp["w2_gs"][0])
    assert rel_err(got, dense_swiglu(x, w1, w2, H)) < 1e-12


def test_global_scales_are_exact_factors():
    inp = wl.make_custom(T=20, D=64, H=64, E=3, k=2, seed=52, routing="uniform", dtype="nvfp4")
    base = run(inp, act=oracle.ACT_EXACT)
    # W2's global scale multiplies each expert's output: x2 on every expert -> x2 exactly
    doubled = run(dict(inp, w2_gs=inp["w2_gs"] * np.float32(2)), act=oracle.ACT_EXACT)
    assert np.array_equal(doubled, 2.0 * base)
    # only x_gs * w1_gs enters GEMM1: moving a factor 2 between them changes nothing
    moved = run(dict(inp, x_gs=np.float32(inp["x_gs"] * 2), w1_gs=inp["w1_gs"] * np.float32(0.5)),
                act=oracle.ACT_EXACT)
    assert np.array_equal(moved, base)
    # a per-expert global scale acts on that expert alone
    gs = inp["w2_gs"].copy()
    gs[1] = 0.0
    ids = inp["topk_ids"]
    alone = run(dict(inp, w2_gs=gs), act=oracle.ACT_EXACT)
    untouched = ~(ids == 1).any(axis=1)
    assert np.array_equal(alone[untouched], base[untouched])
    assert not np.array_equal(alone[~untouched], base[~untouched])


def test_act_requantization_matches_generator_encoder():
    """act requantized per 16 along H with a global scale: the generator's
    encoder applied to the fp32 act gives the same values up to decisions at
    rounding boundaries (fp64 act against its binary32 rounding)."""
    T, D, H = 10, 64, 96
    inp = wl.make_custom(T=T, D=D, H=H, E=1, k=1, seed=53, routing="uniform", dtype="nvfp4")
    inp["topk_w"] = np.ones((T, 1), np.float32)
    x = decode_nv4(inp["x"], inp["x_sf"], inp["x_gs"])
    w1 = decode_nv4(inp["w1"][0], inp["w1_sf"][0], inp["w1_gs"][0])
    w2 = decode_nv4(inp["w2"][0], inp["w2_sf"][0], inp["w2_gs"][0])
    g, u = x @ w1[:H].T, x @ w1[H:].T
    a = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
    act_gs = wl.nv4_global_scale(a)
    packed, sf = wl.nv4_encode_rows(a, act_gs)
    ref = decode_nv4(packed, sf, act_gs) @ w2.T
    got = run(inp, act=oracle.ACT_NVFP4, act_gs=float(act_gs))
    assert rel_err(got, ref) < 1e-6
    exact = run(inp, act=oracle.ACT_EXACT)
    assert 1e-2 < rel_err(got, exact) < 0.5          # 4-bit requantization really happened


def test_equals_mxfp8_mode_on_shared_values():
    """NVFP4 operands whose two 16-blocks of every 32-block carry the same
    power-of-two scale, with global scales 1, are MXFP8 operands (E2M1 values
    are e4m3 values, 2^k is both an e4m3 and an e8m0 scale): both oracle modes
    must agree bit for bit, for several experts and k > 1."""
    rng = np.random.default_rng(54)
    T, D, H, E, k = 12, 64, 64, 4, 2

    def operand(shape):
        rows, cols = int(np.prod(shape[:-1])), shape[-1]
        packed = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
        ex = rng.integers(-8, 1, (rows, cols // 32))
        sf_nv = np.repeat(torch.from_numpy(np.ldexp(1.0, ex).astype(np.float32)).to(torch.float8_e4m3fn)
                          .view(torch.uint8).numpy(), 2, axis=1)
        codes8 = torch.from_numpy(unpack(packed).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        sf_mx = (ex + 127).astype(np.uint8)
        return (packed.reshape(shape[:-1] + (cols // 2,)), sf_nv.reshape(shape[:-1] + (cols // 16,)),
                codes8.reshape(shape), sf_mx.reshape(shape[:-1] + (cols // 32,)))

    x4, xsf4, x8, xsf8 = operand((T, D))
    a4, asf4, a8, asf8 = operand((E, 2 * H, D))
    b4, bsf4, b8, bsf8 = operand((E, D, H))
    ids = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    tw = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    ones = np.ones(E, np.float32)
    nv = oracle.moe_ffn_nvfp4(x4, xsf4, 1.0, a4, asf4, ones, b4, bsf4, ones, ids, tw, act=oracle.ACT_EXACT)
    mx = oracle.moe_ffn(x8, a8, b8, ids, tw, act=oracle.ACT_EXACT, x_sf=xsf8, w1_sf=asf8, w2_sf=bsf8)
    assert np.array_equal(nv, mx)


def test_bad_arguments_rejected():
    inp = wl.make_custom(T=4, D=64, H=64, E=2, k=1, seed=55, routing="uniform", dtype="nvfp4")
    bad = dict(inp, topk_ids=np.full((4, 1), 2, np.int32))
    try:
        run(bad)
        raise AssertionError("an expert id outside [0, E) was accepted")
    except ValueError:
        pass
    try:
        run(inp, act=oracle.ACT_NVFP4, act_gs=0.0)
        raise AssertionError("a zero act global scale was accepted")
    except ValueError:
        pass


def test_clamp_and_bf16_act_on_decoded_operands():
    """The clamped SwiGLU and the bf16-rounded act of the NVFP4 mode against a
    dense computation on operands decoded here (one expert, top-1)."""
    T, D, H = 6, 64, 64
    inp = wl.make_custom(T=T, D=D, H=H, E=1, k=1, seed=56, routing="uniform", dtype="nvfp4")
    inp["topk_w"] = np.ones((T, 1), np.float32)
    x = decode_nv4(inp["x"], inp["x_sf"], inp["x_gs"])
    w1 = decode_nv4(inp["w1"][0], inp["w1_sf"][0], inp["w1_gs"][0])
    w2 = decode_nv4(inp["w2"][0], inp["w2_sf"][0], inp["w2_gs"][0])
    g, u = x @ w1[:H].T, x @ w1[H:].T
    lim = float(np.quantile(np.abs(np.concatenate([g.ravel(), u.ravel()])), 0.5))
    gc, uc = np.minimum(g, lim), np.clip(u, -lim, lim)
    ref = (gc / (1.0 + np.exp(-gc)) * uc) @ w2.T
    got = run(inp, act=oracle.ACT_EXACT, swiglu_limit=lim)
    assert rel_err(got, ref) < 1e-12
    assert rel_err(run(inp, act=oracle.ACT_EXACT), ref) > 1e-3          # the clamp was active
    a = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
    a_bf16 = torch.from_numpy(a).to(torch.bfloat16).double().numpy()
    assert rel_err(run(inp, act=oracle.ACT_BF16), a_bf16 @ w2.T) < 1e-12
