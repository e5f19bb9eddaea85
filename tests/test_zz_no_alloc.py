"""The allocation-free routing entry point (for callers that cannot allocate
device memory: its scratch is a fixed array inside the library) gives the same
counts, offsets and slot permutation as moe_ffn_route with a caller
workspace, on two calls in a row.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import grouped_gemm_gb300 as moe
from grouped_gemm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def with_workspace(ids, tw, E):
    T, k = ids.shape
    ws = moe.alloc_workspace(T, E, 128, 128, k, moe.MOE_BF16, moe.MOE_FUSED)
    c = torch.empty(E, dtype=torch.int32, device="cuda")
    o = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    s = torch.empty(T * k, dtype=torch.int32, device="cuda")
    moe.moe_ffn_route(ids, tw, T, E, k, c, o, s, ws)
    assert moe.moe_ffn_sync_status(ws) == 0
    return c.cpu(), o.cpu(), s.cpu()


def without_workspace(ids, tw, E):
    T, k = ids.shape
    c = torch.full((E,), -5, dtype=torch.int32, device="cuda")
    o = torch.full((E + 1,), -5, dtype=torch.int32, device="cuda")
    s = torch.full((T * k,), -5, dtype=torch.int32, device="cuda")
    bits = torch.full((1,), -5, dtype=torch.int32, device="cuda")
    # straight through the C ABI
    st = moe.lib().moe_ffn_route_noalloc(ids.data_ptr(), tw.data_ptr(), T, E, k, c.data_ptr(), o.data_ptr(),
                                         s.data_ptr(), bits.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, moe.moe_ffn_status_string(st)
    torch.cuda.synchronize()
    return c.cpu(), o.cpu(), s.cpu(), int(bits.item())


@pytest.mark.parametrize("name", ["prefill", "decode"])
def test_noalloc_route_matches_workspace_route_twice(name):
    w = wl.WORKLOADS[name]
    rng = np.random.default_rng(42)
    ids_np, tw_np = wl.draw_routing(rng, w.T, w.E, w.k, w.routing)
    ids = torch.from_numpy(ids_np).cuda()
    tw = torch.from_numpy(tw_np).cuda()
    ref = with_workspace(ids, tw, w.E)
    for _ in range(2):
        got = without_workspace(ids, tw, w.E)
        assert got[3] == 0
        for a, b in zip(got[:3], ref):
            assert torch.equal(a, b)


def test_noalloc_route_second_problem_after_first():
    # a different, smaller problem right after a larger one: stale scratch
    # contents from the previous call must not leak into the result
    rng = np.random.default_rng(5)
    for T, E, k in ((4096, 128, 8), (33, 5, 3)):
        ids_np, tw_np = wl.draw_routing(rng, T, E, k, "uniform")
        ids, tw = torch.from_numpy(ids_np).cuda(), torch.from_numpy(tw_np).cuda()
        ref = with_workspace(ids, tw, E)
        got = without_workspace(ids, tw, E)
        for a, b in zip(got[:3], ref):
            assert torch.equal(a, b)


def test_noalloc_route_reports_bad_ids_and_rejects_oversize():
    ids = torch.zeros(10, 2, dtype=torch.int32, device="cuda")
    ids[3, 1] = 77
    tw = torch.ones(10, 2, device="cuda")
    c, o, s, bits = without_workspace(ids, tw, 8)
    assert bits == 1 and int(c.sum()) == 19 and int(s[7]) == -1
    # the next good call starts with clean status words
    c, o, s, bits = without_workspace(torch.zeros(10, 2, dtype=torch.int32, device="cuda"), tw, 8)
    assert bits == 0 and int(c[0]) == 20
    big = torch.zeros(131072 // 8 + 1, 8, dtype=torch.int32, device="cuda")
    st = moe.moe_ffn_route_noalloc(big, torch.ones_like(big, dtype=torch.float32), big.shape[0], 8, 8, None, None,
                                   None, check=False)
    assert st == 5  # MOE_ERR_WORKSPACE_TOO_SMALL
