"""Pins for the oracle's MXFP4 weight mode: E2M1 elements (OCP Microscaling
Formats: 1 sign, 2 exponent bits with bias 1, 1 mantissa bit, no Inf/NaN) with
one e8m0 scale per 32 elements, weights packed two codes to a byte: the
routed-weight format of "GC-MoE on SM120" (sec. 2.2, scale formats), run
there against MXFP8 (E4M3) activations.  Each test checks the oracle against something other
than itself: the format's 16-value table, brute-force nearest rounding, the
input generator's independent numpy encoder, and a dense fp64 SwiGLU FFN on
weights decoded here from that table.  CPU only."""
import numpy as np
import torch

import oracle
from grouped_gemm_gb300 import workloads as wl

# OCP E2M1 values of codes 0..15 (sign in bit 3)
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def decode_fp4(packed, sf):
    """Test-side decode: table lookup, low nibble first, times 2^(sf-127)."""
    tab = np.array(E2M1_TABLE)
    lo = tab[packed & 0xF]
    hi = tab[packed >> 4]
    v = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,))
    v[..., 0::2] = lo
    v[..., 1::2] = hi
    return v * np.repeat(np.ldexp(1.0, sf.astype(np.int64) - 127), 32, axis=-1)


def decode_fp8(q, sf):
    v = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
    return v * np.repeat(np.ldexp(1.0, sf.astype(np.int64) - 127), 32, axis=-1)


def rel_err(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


def test_e2m1_decode_matches_ocp_table():
    got = oracle.e2m1_to_f64(np.arange(16, dtype=np.uint8))
    assert got.tolist() == E2M1_TABLE
    assert np.array_equal(np.signbit(got), np.signbit(np.array(E2M1_TABLE)))


def test_e2m1_encode_roundtrip_and_ties():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(oracle.f64_to_e2m1(np.array(E2M1_TABLE)), codes)
    # midpoints go to the code with mantissa bit 0
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    want = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    got = oracle.e2m1_to_f64(oracle.f64_to_e2m1(np.array(mids)))
    assert got.tolist() == want
    got = oracle.e2m1_to_f64(oracle.f64_to_e2m1(-np.array(mids)))
    assert got.tolist() == [-v for v in want]
    # saturation to +-6
    assert oracle.e2m1_to_f64(oracle.f64_to_e2m1(np.array([6.0, 6.5, 7.0, 1e30, -1e30]))).tolist() == \
        [6.0, 6.0, 6.0, 6.0, -6.0]


def test_e2m1_encode_is_nearest_brute_force():
    rng = np.random.default_rng(40)
    v = np.concatenate([rng.uniform(-7, 7, 20000), rng.uniform(-1, 1, 5000)])
    got = oracle.e2m1_to_f64(oracle.f64_to_e2m1(v))
    grid = np.array(E2M1_TABLE[:8])
    a = np.minimum(np.abs(v), 6.0)
    d = np.abs(a[:, None] - grid[None, :])
    nearest = grid[np.argmin(d, axis=1)]
    tie = (np.sort(d, axis=1)[:, 1] == d.min(axis=1))
    assert not tie.any()                        # random draws: no exact midpoints
    assert np.array_equal(np.abs(got), nearest)
    assert np.array_equal(np.sign(got[got != 0]), np.sign(v[got != 0]))


def test_mx4_scale_exponent_is_smallest_nonsaturating_power():
    rng = np.random.default_rng(41)
    amaxes = np.concatenate([rng.uniform(1e-3, 1e3, 2000), 6.0 * np.ldexp(1.0, np.arange(-10, 10)),
                             np.ldexp(1.0, np.arange(-10, 10)), 1.5 * np.ldexp(1.0, np.arange(-10, 10))])
    for amax in amaxes:
        e = oracle.mx4_scale_exponent(float(amax))
        assert amax * 2.0 ** -e <= 6.0 < amax * 2.0 ** -(e - 1)
    assert oracle.mx4_scale_exponent(0.0) == 0


def test_generator_encoder_agrees_with_oracle_codec():
    """The input generator's numpy encoder and the oracle's C codec are written
    separately; they must choose the same scale and the same code everywhere."""
    rng = np.random.default_rng(42)
    a = (rng.standard_normal((64, 256)) * 10.0 ** rng.integers(-3, 3, (64, 1))).astype(np.float32)
    packed, sf = wl.mx4_encode_rows(a)
    blk = a.reshape(-1, 32).astype(np.float64)
    e = np.array([oracle.mx4_scale_exponent(float(m)) for m in np.abs(blk).max(1)])
    assert np.array_equal(sf.reshape(-1).astype(np.int64) - 127, e)
    codes = oracle.f64_to_e2m1(blk * np.ldexp(1.0, -e)[:, None]).reshape(a.shape)
    assert np.array_equal(packed, (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8))
    # each dequantized element is within half a grid step (at most 1 x 2^e) of its input
    deq = decode_fp4(packed, sf).reshape(-1, 32)
    assert (np.abs(deq - np.clip(blk, -6 * np.ldexp(1.0, e)[:, None], 6 * np.ldexp(1.0, e)[:, None]))
            <= np.ldexp(1.0, e)[:, None]).all()


def dense_swiglu(x, w1, w2, H):
    g = x @ w1[:H].T
    u = x @ w1[H:].T
    return (g / (1.0 + np.exp(-g)) * u) @ w2.T


def test_fp4_weights_dense_single_expert():
    """top-1 with weight 1 over one expert is that expert's dense SwiGLU FFN on
    the decoded weights (x MXFP8, exact act)."""
    T, D, H = 9, 64, 96
    inp = wl.make_custom(T=T, D=D, H=H, E=1, k=1, seed=43, routing="uniform", dtype="mxfp4w")
    ones = np.ones((T, 1), np.float32)
    got = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], ones, act=oracle.ACT_EXACT,
                         x_sf=inp["x_sf"], w1_sf=inp["w1_sf"], w2_sf=inp["w2_sf"], fp4_weights=True)
    x = decode_fp8(inp["x"], inp["x_sf"])
    ref = dense_swiglu(x, decode_fp4(inp["w1"][0], inp["w1_sf"][0]), decode_fp4(inp["w2"][0], inp["w2_sf"][0]), H)
    assert rel_err(got, ref) < 1e-12


def test_fp4_nibble_order():
    """A single nonzero weight at an odd element sits in a byte's high nibble:
    moving it to the low nibble must move the contribution to the even input."""
    T, D, H = 2, 64, 32
    x = np.zeros((T, D), np.float64)
    x[0, 5], x[1, 4] = 1.0, 1.0                                  # token 0 sees column 5, token 1 column 4
    xq = oracle.f64_to_e4m3(x)
    x_sf = np.full((T, D // 32), 127, np.uint8)
    w1 = np.zeros((1, 2 * H, D // 2), np.uint8)
    w1[0, 0, 2] = 0x2 << 4                                        # gate[0] = 1.0 * x[5]
    w1[0, H, 2] = 0x4 << 4                                        # up[0]   = 2.0 * x[5]
    w1_sf = np.full((1, 2 * H, D // 32), 127, np.uint8)
    w2 = np.zeros((1, D, H // 2), np.uint8)
    w2[0, 3, 0] = 0x2                                             # out[3] = 1.0 * act[0]  (low nibble)
    w2_sf = np.full((1, D, H // 32), 127, np.uint8)
    ids = np.zeros((T, 1), np.int32)
    tw = np.ones((T, 1), np.float32)
    got = oracle.moe_ffn(xq, w1, w2, ids, tw, act=oracle.ACT_EXACT, x_sf=x_sf, w1_sf=w1_sf, w2_sf=w2_sf,
                         fp4_weights=True)
    want0 = 1.0 / (1.0 + np.exp(-1.0)) * 2.0
    assert abs(got[0, 3] - want0) < 1e-15 and np.count_nonzero(got[0]) == 1
    assert not got[1].any()


def test_fp4_mode_equals_fp8_mode_on_shared_values():
    """Every E2M1 value is an e4m3 value, so the same weights re-coded as MXFP8
    (same scales) must give bit-identical oracle outputs through the MXFP8 path,
    for several experts, k > 1 and the bf16-rounded act."""
    T, D, H, E, k = 24, 64, 64, 4, 2
    inp = wl.make_custom(T=T, D=D, H=H, E=E, k=k, seed=44, routing="uniform", dtype="mxfp4w")
    tab = np.array(E2M1_TABLE)

    def to_fp8(packed):
        v = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,))
        v[..., 0::2] = tab[packed & 0xF]
        v[..., 1::2] = tab[packed >> 4]
        q = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy(), v)
        return q

    for act in (oracle.ACT_EXACT, oracle.ACT_BF16, oracle.ACT_MXFP8):
        a = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=act,
                           x_sf=inp["x_sf"], w1_sf=inp["w1_sf"], w2_sf=inp["w2_sf"], fp4_weights=True)
        b = oracle.moe_ffn(inp["x"], to_fp8(inp["w1"]), to_fp8(inp["w2"]), inp["topk_ids"], inp["topk_w"], act=act,
                           x_sf=inp["x_sf"], w1_sf=inp["w1_sf"], w2_sf=inp["w2_sf"])
        assert np.array_equal(a, b)
