"""Routing permutation on the GPU is bit-exact against the oracle's counting
sort ("Prime Flash MoE" sec. 3 and 6: tokens processed in per-expert sorted
order), including empty experts, one hot expert, repeats and T = 1.  Problems
too large for the single-block kernel run both through the one-launch
cooperative routing (default) and the three-launch path, with 256 tokens per
routing block and with fewer (64, 128); the single-block
kernel is also run on every problem it can take (at most 256 experts) with
its size limit raised."""
import numpy as np
import pytest
import torch

import grouped_gemm_gb300 as moe
import oracle
from grouped_gemm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=[(1, 8192, 0), (0, 8192, 0), (1, 1 << 20, 0), (1, 8192, 64), (0, 8192, 128)],
                ids=["coop", "three_launches", "single_block", "coop_tpb64", "three_launches_tpb128"])
def route_mode(request):
    coop, small_pairs, tpb = request.param
    moe.moe_ffn_set_option(moe.MOE_OPT_ROUTE_COOP, coop)
    moe.moe_ffn_set_option(moe.MOE_OPT_ROUTE_SMALL_PAIRS, small_pairs)
    moe.moe_ffn_set_option(moe.MOE_OPT_ROUTE_TPB, tpb)  # tokens per routing block (0: 256)
    yield request.param
    moe.moe_ffn_set_option(moe.MOE_OPT_ROUTE_COOP, 1)
    moe.moe_ffn_set_option(moe.MOE_OPT_ROUTE_SMALL_PAIRS, 8192)
    moe.moe_ffn_set_option(moe.MOE_OPT_ROUTE_TPB, 0)


def gpu_route(ids, E):
    T, k = ids.shape
    dev_ids = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda()
    dev_w = torch.rand(T, k, device="cuda")
    ws = moe.alloc_workspace(max(T, 1), E, 128, 128, k, moe.MOE_BF16, moe.MOE_FUSED)
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    slot = torch.full((max(T * k, 1),), -7, dtype=torch.int32, device="cuda")
    moe.moe_ffn_route(dev_ids, dev_w, T, E, k, counts, offsets, slot, ws)
    st = moe.moe_ffn_sync_status(ws)
    return st, counts.cpu().numpy(), offsets.cpu().numpy(), slot.cpu().numpy()[:T * k]


def expected_padded(ref, ids, w, E):
    """The padded tables the GEMMs read, from the oracle's padded offsets and
    padded slot of every pair: row_tok / slot_w of each padded slot, the expert
    of each 128-row block, and pairs of consecutive blocks of one expert."""
    T, k = ids.shape
    po = ref["pad_offsets"]
    s_pad = int(po[E])
    row_tok = np.full(s_pad, -1, np.int64)
    slot_w = np.zeros(s_pad, np.float32)
    ps = ref["pad_slot_of_pair"]
    row_tok[ps] = np.arange(T * k) // k
    slot_w[ps] = w.ravel()
    nrb = (po[1:] - po[:-1]) // 128
    expert_of_rb = np.repeat(np.arange(E), nrb)
    pairs = []
    for e in range(E):
        rb0 = int(po[e]) // 128
        for q in range(0, int(nrb[e]), 2):
            pairs.append(((rb0 + q) << 1) | (1 if q + 1 < nrb[e] else 0))
    return dict(row_tok=row_tok, slot_w=slot_w, expert_of_rb=expert_of_rb, pair_info=np.array(pairs, np.int64),
                n_blocks=s_pad // 128)


def check_padded(ids, E, ref):
    """moe_ffn_route_padded against the oracle, bit for bit (slot_w compared as
    float32 bit patterns: each is a copied routing weight)."""
    T, k = ids.shape
    rng = np.random.default_rng(T * 7 + E)
    w = rng.random((T, k), dtype=np.float32)
    smax = moe.moe_ffn_route_padded_slots(T, E, k)
    dev_ids = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda()
    ws = moe.alloc_workspace(T, E, 128, 128, k, moe.MOE_BF16, moe.MOE_FUSED)
    fill = lambda n, dt=torch.int32: torch.full((n,), -7, dtype=dt, device="cuda")
    po, erb, pinfo = fill(E + 1), fill(smax // 128), fill(smax // 128)
    rtok, sw, nb = fill(smax), torch.full((smax,), -7.0, device="cuda"), fill(2)
    moe.moe_ffn_route_padded(dev_ids, torch.from_numpy(w).cuda(), T, E, k, po, erb, pinfo, rtok, sw, nb, ws)
    assert moe.moe_ffn_sync_status(ws) == 0
    exp = expected_padded(ref, ids, w, E)
    n_rb, n_pairs = (int(v) for v in nb.cpu().numpy())
    assert np.array_equal(po.cpu().numpy(), ref["pad_offsets"])
    assert n_rb == exp["n_blocks"] and n_pairs == exp["pair_info"].size
    assert np.array_equal(erb.cpu().numpy()[:n_rb], exp["expert_of_rb"])
    assert np.array_equal(pinfo.cpu().numpy()[:n_pairs], exp["pair_info"])
    s_pad = n_rb * 128
    assert np.array_equal(rtok.cpu().numpy()[:s_pad], exp["row_tok"])
    assert np.array_equal(sw.cpu().numpy()[:s_pad].view(np.uint32), exp["slot_w"].view(np.uint32))


def check(ids, E):
    st, c, o, s = gpu_route(ids, E)
    assert st == 0
    ref = oracle.route(ids, E)
    assert np.array_equal(c, ref["counts"])
    assert np.array_equal(o, ref["offsets"])
    assert np.array_equal(s, ref["slot_of_pair"])
    if ids.shape[0] > 0:
        check_padded(ids, E, ref)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "mxfp8"])
def test_route_workloads(name):
    w = wl.WORKLOADS[name]
    ids, _ = wl.draw_routing(np.random.default_rng(0), w.T, w.E, w.k, w.routing)
    check(ids, w.E)


def test_route_large_skewed():
    w = wl.WORKLOADS["large_skewed"]
    ids, _ = wl.draw_routing(np.random.default_rng(0), w.T, w.E, w.k, "zipf")
    ref = oracle.route(ids, w.E)
    assert (ref["counts"] == 0).sum() == 8          # the zero-popularity experts
    check(ids, w.E)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (1, 8, 8), (3, 1024, 4), (777, 5, 3), (513, 300, 2), (9000, 1, 1),
                                   (20000, 1024, 8), (65536, 7, 1), (4097, 128, 8)])
def test_route_shapes(T, E, k):
    ids, _ = wl.draw_routing(np.random.default_rng(T), T, E, k, "uniform") if k <= E else (None, None)
    check(ids, E)


def test_route_all_on_one_expert_and_repeats():
    rng = np.random.default_rng(3)
    check(np.full((1000, 4), 5, np.int32), 16)
    check(rng.integers(0, 3, size=(2049, 8)).astype(np.int32), 7)


def test_route_bad_id_reported():
    ids = np.zeros((10, 2), np.int32)
    ids[4, 1] = 9
    st, c, _, s = gpu_route(ids, 8)
    assert st == 4  # MOE_ERR_BAD_ROUTING
    assert c.sum() == 19 and s[9] == -1


def test_route_bad_id_reported_multi_block():
    rng = np.random.default_rng(9)
    ids = rng.integers(0, 16, size=(6000, 2)).astype(np.int32)
    ids[4321, 0] = -3
    st, c, _, s = gpu_route(ids, 16)
    assert st == 4  # MOE_ERR_BAD_ROUTING
    assert c.sum() == 6000 * 2 - 1 and s[4321 * 2] == -1
    ref = oracle.route(np.where(ids < 0, 0, ids), 16)
    assert c[0] == ref["counts"][0] - 1
