"""Routing permutation on the GPU is bit-exact against the oracle's counting
sort ("Prime Flash MoE" sec. 3 and 6: tokens processed in per-expert sorted
order), including empty experts, one hot expert, repeats and T = 1.  Problems
too large for the single-block kernel run both through the one-launch
cooperative routing (default) and the three-launch path."""
import numpy as np
import pytest
import torch

import grouped_gemm_gb300 as moe
import oracle
from grouped_gemm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=[1, 0], ids=["coop", "three_launches"])
def route_mode(request):
    moe.moe_ffn_set_option(moe.MOE_OPT_ROUTE_COOP, request.param)
    yield request.param
    moe.moe_ffn_set_option(moe.MOE_OPT_ROUTE_COOP, 1)


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


def check(ids, E):
    st, c, o, s = gpu_route(ids, E)
    assert st == 0
    ref = oracle.route(ids, E)
    assert np.array_equal(c, ref["counts"])
    assert np.array_equal(o, ref["offsets"])
    assert np.array_equal(s, ref["slot_of_pair"])


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill"])
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
