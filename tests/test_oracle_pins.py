"""Pins for the CPU oracle: each test checks it against something other than
itself -- a library routine, a closed form, brute force or an invariant of the
method ("Prime Flash MoE - Faster MoE Kernels optimized for Blackwell", sec. 1
"The computation"; invariants of the method: top-1 with weight 1 is the dense
SwiGLU FFN of that expert, identical experts scale by the weight sum, token
order does not matter).  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
from grouped_gemm_gb300 import workloads as wl


def bf16_bits_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def f64_to_bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float64)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


# ----------------------------------------------------------------- formats
def test_bf16_decode_all_patterns_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f64(bits)
    ref = bf16_bits_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_f32_to_bf16_rne_matches_torch():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32),
        # exact ties between two bf16 values: low 16 bits == 0x8000
        (rng.integers(0, 2**31, 4000, dtype=np.int64).astype(np.uint32) & 0xFFFF0000 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 3.3895314e38, 3.4e38, 1e-40, -1e-45], np.float32),
    ])
    v = v[np.isfinite(v)]
    ours = oracle.f32_to_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_e4m3_decode_all_codes_matches_torch_and_ocp_table():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # OCP MX spec E4M3 table points
    assert ours[0x7E] == 448.0 and ours[0xFE] == -448.0
    assert ours[0x08] == 2.0 ** -6 and ours[0x01] == 2.0 ** -9 and ours[0x07] == 7 * 2.0 ** -9
    assert ours[0x38] == 1.0
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF]) and nan.sum() == 2


def test_e4m3_encode_rne_matches_torch_in_range():
    rng = np.random.default_rng(2)
    finite = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = (finite[:-1] + finite[1:]) / 2                       # exact ties
    v = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(5000) * 0.01, mids, -mids])
    ours = oracle.f64_to_e4m3(v)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # -0.0 vs +0.0 codes may differ in sign only for exact zeros
    assert np.array_equal(ours, ref)


def test_e4m3_encode_saturates():
    assert oracle.f64_to_e4m3(np.array([448.0, 460.0, 1e9, -1e9]))[:].tolist() == [0x7E, 0x7E, 0x7E, 0xFE]
    assert oracle.f64_to_e4m3(np.array([464.0]))[0] == 0x7E     # would round to 512 without satfinite


def test_mx_scale_exponent_is_smallest_nonsaturating_power():
    rng = np.random.default_rng(3)
    vals = list(rng.lognormal(0, 6, 3000))
    for p in range(-20, 20):
        vals += [1.75 * 2.0 ** p, np.nextafter(1.75 * 2.0 ** p, 10.0), np.nextafter(1.75 * 2.0 ** p, 0.0), 2.0 ** p]
    for amax in vals:
        e = oracle.mx_scale_exponent(amax)
        # brute force: smallest integer e with amax * 2^-e <= 448
        eb = -200
        while amax * 2.0 ** (-eb) > 448.0:
            eb += 1
        assert e == eb, amax
    assert oracle.mx_scale_exponent(0.0) == 0


def test_mx_quantize_block_properties():
    rng = np.random.default_rng(4)
    a = rng.standard_normal(32 * 400) * np.exp(rng.uniform(-8, 8, 400)).repeat(32)
    a[:32] = 0.0
    q, sf, deq = oracle.mx_quantize(a)
    assert sf[0] == 127 and not q[:32].any()
    dec = oracle.e4m3_to_f64(q).reshape(-1, 32)
    # before rounding, each block's amax lands in (224, 448]; after e4m3
    # rounding it can touch 224 (the grid step there is 16)
    blk = a.astype(np.float32).astype(np.float64).reshape(-1, 32)[1:]
    pre = np.abs(blk).max(axis=1) * np.ldexp(1.0, 127 - sf[1:].astype(int))
    assert (pre > 224).all() and (pre <= 448).all()
    scaled_max = np.abs(dec).max(axis=1)[1:]
    assert (scaled_max >= 224).all() and (scaled_max <= 448).all()
    # dequantized = code * 2^(sf-127), within half an e4m3 step of the input
    assert np.array_equal(deq.reshape(-1, 32), dec * np.ldexp(1.0, sf.astype(int) - 127)[:, None])
    rel = np.abs(deq - a.astype(np.float32)) / np.maximum(np.abs(a), 1e-300)
    big = np.abs(a) > np.repeat(np.abs(a).reshape(-1, 32).max(1), 32) * 2.0 ** -6
    assert rel[big].max() <= 2.0 ** -4 + 1e-12
    # the generator's independent encoder (numpy + torch cast) agrees exactly
    gq, gsf = wl.mx_encode_rows(a.astype(np.float32).reshape(-1, 32))
    assert np.array_equal(gq.ravel(), q) and np.array_equal(gsf.ravel(), sf)


# ----------------------------------------------------------------- routing
@pytest.mark.parametrize("T,E,k,kind", [(64, 8, 2, "topk_logits"), (1, 4, 4, "uniform"), (300, 16, 8, "zipf"),
                                        (0, 4, 2, "uniform"), (257, 128, 8, "zipf")])
def test_route_matches_brute_force(T, E, k, kind):
    rng = np.random.default_rng(5)
    ids, _ = wl.draw_routing(rng, T, E, k, kind) if T else (np.zeros((0, k), np.int32), None)
    r = oracle.route(ids, E)
    flat = ids.ravel()
    counts = np.array([(flat == e).sum() for e in range(E)])
    assert np.array_equal(r["counts"], counts)
    assert r["offsets"][0] == 0 and np.array_equal(np.diff(r["offsets"]), counts)
    # brute force: a stable sort by expert id gives the pair in each slot
    order = np.argsort(flat, kind="stable")
    slot = np.empty_like(order)
    slot[order] = np.arange(flat.size)
    assert np.array_equal(r["slot_of_pair"], slot)
    # bijection, stability within each expert
    assert np.array_equal(np.sort(r["slot_of_pair"]), np.arange(flat.size))
    for e in range(E):
        s = r["slot_of_pair"][flat == e]
        assert (np.diff(s) > 0).all()
    padc = (counts + 127) // 128 * 128
    assert np.array_equal(np.diff(r["pad_offsets"]), padc)
    assert np.array_equal(r["pad_slot_of_pair"] - r["pad_offsets"][flat], r["slot_of_pair"] - r["offsets"][flat])


def test_route_duplicate_ids_and_empty_experts():
    ids = np.array([[3, 3], [0, 3], [3, 0]], np.int32)
    r = oracle.route(ids, 6)
    assert r["counts"].tolist() == [2, 0, 0, 4, 0, 0]
    assert r["slot_of_pair"].tolist() == [2, 3, 0, 4, 5, 1]
    assert r["pad_offsets"].tolist() == [0, 128, 128, 128, 256, 256, 256]


def test_route_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.route(np.array([[0, 4]], np.int32), 4)
    with pytest.raises(ValueError):
        oracle.route(np.array([[-1, 0]], np.int32), 4)


# ----------------------------------------------------------------- forward
def dense_ffn_torch(x, w1, w2, H, act_round=None):
    """Library special case: one expert, dense fp64 torch matmuls."""
    g = x @ w1[:H].T
    u = x @ w1[H:].T
    a = torch.nn.functional.silu(g) * u
    if act_round == "bf16":
        a = a.float().to(torch.bfloat16).double()
    return a @ w2.T


def per_expert_loop_torch(x, w1, w2, ids, tw, act_round=None):
    """The pages' naive per-expert loop (sec. 1): for every expert, the FFN of
    the tokens routed to it, weighted and added to their output rows."""
    T, D = x.shape
    E, H2, _ = w1.shape
    out = torch.zeros(T, D, dtype=torch.float64)
    for e in range(E):
        t_idx, j_idx = np.nonzero(ids == e)
        if t_idx.size == 0:
            continue
        y = dense_ffn_torch(x[t_idx], w1[e], w2[e], H2 // 2, act_round)
        out.index_add_(0, torch.from_numpy(t_idx), torch.from_numpy(tw[t_idx, j_idx]).double()[:, None] * y)
    return out.numpy()


def rel_err(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


@pytest.mark.parametrize("act", ["exact", "bf16"])
def test_top1_weight1_is_dense_ffn(act):
    inp = wl.make_custom(T=24, D=64, H=32, E=1, k=1, seed=6)
    x = torch.from_numpy(bf16_bits_to_f64(inp["x"]))
    w1 = torch.from_numpy(bf16_bits_to_f64(inp["w1"][0]))
    w2 = torch.from_numpy(bf16_bits_to_f64(inp["w2"][0]))
    tw = np.ones((24, 1), np.float32)
    mode = oracle.ACT_EXACT if act == "exact" else oracle.ACT_BF16
    ours = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], tw, act=mode)
    ref = dense_ffn_torch(x, w1, w2, 32, act_round=None if act == "exact" else "bf16").numpy()
    assert rel_err(ours, ref) < 1e-12


@pytest.mark.parametrize("T,D,H,E,k,kind", [(64, 256, 128, 8, 2, "topk_logits"), (37, 128, 64, 6, 3, "uniform"),
                                            (50, 64, 32, 16, 4, "zipf")])
def test_matches_per_expert_loop(T, D, H, E, k, kind):
    inp = wl.make_custom(T=T, D=D, H=H, E=E, k=k, seed=7, routing=kind)
    x = torch.from_numpy(bf16_bits_to_f64(inp["x"]))
    w1 = torch.from_numpy(bf16_bits_to_f64(inp["w1"]))
    w2 = torch.from_numpy(bf16_bits_to_f64(inp["w2"]))
    for mode, ar in ((oracle.ACT_EXACT, None), (oracle.ACT_BF16, "bf16")):
        ours = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=mode)
        ref = per_expert_loop_torch(x, w1, w2, inp["topk_ids"], inp["topk_w"], ar)
        assert rel_err(ours, ref) < 1e-12
    # selected tokens only
    sel = np.array([5, 0, T - 1], np.int32)
    part = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], tokens=sel)
    full = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"])
    assert np.array_equal(part, full[sel])


def test_closed_form_permutation_experts():
    """W1 gate = a P1, W1 up = b P2, W2 = c P3 with permutation matrices (D = H):
    out[t, d] = sum_j w_j c silu(a x[p1[p3[d]]]) b x[p2[p3[d]]] -- catches a
    transposed operand, swapped gate/up halves and a wrong sum order."""
    rng = np.random.default_rng(8)
    D = H = 32
    E, k, T = 3, 2, 10
    coef = [(0.5, 1.5, 2.0), (0.25, -1.0, 0.5), (1.0, 0.75, -1.5)]
    perms = [[rng.permutation(D) for _ in range(3)] for _ in range(E)]
    w1 = np.zeros((E, 2 * H, D))
    w2 = np.zeros((E, D, H))
    for e in range(E):
        a, b, c = coef[e]
        p1, p2, p3 = perms[e]
        w1[e, np.arange(H), p1] = a           # gate[h] = a x[p1[h]]
        w1[e, H + np.arange(H), p2] = b       # up[h]   = b x[p2[h]]
        w2[e, np.arange(D), p3] = c           # y[d]    = c act[p3[d]]
    xs = rng.integers(-8, 9, size=(T, D)) / 4.0          # exactly representable in bf16
    ids = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    tw = rng.uniform(0.1, 1.0, size=(T, k)).astype(np.float32)
    got = oracle.moe_ffn(f64_to_bf16_bits(xs), f64_to_bf16_bits(w1), f64_to_bf16_bits(w2), ids, tw,
                         act=oracle.ACT_EXACT)
    silu = lambda z: z / (1.0 + math.exp(-z))
    for t in range(T):
        for d in range(D):
            ref = 0.0
            for j in range(k):
                e = ids[t, j]
                a, b, c = coef[e]
                p1, p2, p3 = perms[e]
                h = p3[d]
                ref += float(tw[t, j]) * c * silu(a * xs[t, p1[h]]) * b * xs[t, p2[h]]
            assert abs(got[t, d] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_invariants():
    T, D, H, E, k = 40, 64, 32, 6, 3
    inp = wl.make_custom(T=T, D=D, H=H, E=E, k=k, seed=9, routing="uniform")
    x, w1, w2, ids, tw = inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"]
    base = oracle.moe_ffn(x, w1, w2, ids, tw, act=oracle.ACT_EXACT)
    scale = lambda a, b: rel_err(a, b)
    # identical experts: out = (sum_j w_j) * single-expert FFN
    w1s, w2s = np.repeat(w1[:1], E, 0), np.repeat(w2[:1], E, 0)
    same = oracle.moe_ffn(x, w1s, w2s, ids, tw, act=oracle.ACT_EXACT)
    one = oracle.moe_ffn(x, w1[:1], w2[:1], np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32),
                         act=oracle.ACT_EXACT)
    assert scale(same, tw.astype(np.float64).sum(1, keepdims=True) * one) < 1e-13
    # token order: permuting tokens permutes the output rows exactly
    perm = np.random.default_rng(10).permutation(T)
    pe = oracle.moe_ffn(x[perm], w1, w2, ids[perm], tw[perm], act=oracle.ACT_EXACT)
    assert np.array_equal(pe, base[perm])
    # linearity in the routing weights
    tw2 = (tw * np.float32(0.5)).astype(np.float32)
    assert scale(oracle.moe_ffn(x, w1, w2, ids, tw2, act=oracle.ACT_EXACT), 0.5 * base) < 1e-14
    # relabeling experts together with the ids leaves the output unchanged
    rp = np.random.default_rng(11).permutation(E)
    inv = np.argsort(rp)
    rel = oracle.moe_ffn(x, w1[rp], w2[rp], inv[ids].astype(np.int32), tw, act=oracle.ACT_EXACT)
    assert np.array_equal(rel, base)
    # x = 0 -> 0; zero gate rows -> silu(0) = 0 -> 0
    assert not oracle.moe_ffn(np.zeros_like(x), w1, w2, ids, tw).any()
    w1z = w1.copy()
    w1z[:, :H] = 0
    assert not oracle.moe_ffn(x, w1z, w2, ids, tw).any()
    # order of the k slots of one token does not matter beyond rounding
    rev = oracle.moe_ffn(x, w1, w2, ids[:, ::-1].copy(), tw[:, ::-1].copy(), act=oracle.ACT_EXACT)
    assert scale(rev, base) < 1e-13


def test_mxfp8_inputs_dequantize_exactly():
    inp = wl.make_custom(T=16, D=64, H=64, E=4, k=2, seed=12, routing="uniform", dtype="mxfp8")

    def deq(q, sf):
        v = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
        s = np.ldexp(1.0, sf.astype(np.int64) - 127)
        return v * np.repeat(s, 32, axis=-1)

    x, w1, w2 = deq(inp["x"], inp["x_sf"]), deq(inp["w1"], inp["w1_sf"]), deq(inp["w2"], inp["w2_sf"])
    got = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_EXACT,
                         x_sf=inp["x_sf"], w1_sf=inp["w1_sf"], w2_sf=inp["w2_sf"])
    ref = per_expert_loop_torch(torch.from_numpy(x), torch.from_numpy(w1), torch.from_numpy(w2), inp["topk_ids"],
                                inp["topk_w"])
    assert rel_err(got, ref) < 1e-12


def test_mxfp8_act_requantization():
    """act requantized per 32 along H: compare with the generator's independent
    encoder (numpy exponent + torch e4m3 cast) applied to the fp32 act."""
    T, D, H, E = 12, 64, 96, 1
    inp = wl.make_custom(T=T, D=D, H=H, E=E, k=1, seed=13, routing="uniform")
    x = torch.from_numpy(bf16_bits_to_f64(inp["x"]))
    w1 = torch.from_numpy(bf16_bits_to_f64(inp["w1"][0]))
    w2 = torch.from_numpy(bf16_bits_to_f64(inp["w2"][0]))
    a = (torch.nn.functional.silu(x @ w1[:H].T) * (x @ w1[H:].T)).numpy().astype(np.float32)
    q, sf = wl.mx_encode_rows(a)
    adq = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy() * np.repeat(
        np.ldexp(1.0, sf.astype(np.int64) - 127), 32, axis=-1)
    ref = adq @ w2.numpy().T
    got = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], np.ones((T, 1), np.float32),
                         act=oracle.ACT_MXFP8)
    # identical quantization decisions except where fp64 vs fp32 act straddles a
    # rounding boundary; those move one code by one step
    assert rel_err(got, ref) < 1e-3
    exact = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], np.ones((T, 1), np.float32),
                           act=oracle.ACT_EXACT)
    assert 1e-3 < rel_err(got, exact) < 0.1      # requantization really happened


def test_bad_ids_rejected():
    inp = wl.make_custom(T=4, D=32, H=32, E=2, k=1, seed=14)
    ids = inp["topk_ids"].copy()
    ids[2, 0] = 2
    with pytest.raises(ValueError):
        oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], ids, inp["topk_w"])
