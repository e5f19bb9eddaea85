"""The C-ABI library loads on a machine without a GPU, exports every entry
point include/moe_ffn.h declares, and rejects bad arguments on the host."""
import ctypes
import os
import re

import pytest

import grouped_gemm_gb300 as moe

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_ffn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("moe_ffn_forward", "moe_ffn_workspace_size", "moe_ffn_route", "moe_ffn_sync_status",
              "moe_ffn_status_string", "moe_ffn_workspace_init", "moe_ffn_set_wait_limit_ns"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(moe.lib()._name)  # rebuilt first if a source is newer
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    for s in range(8):
        assert moe.moe_ffn_status_string(s) and moe.moe_ffn_status_string(s) != "unknown status"


def test_workspace_size_rules():
    ok = moe.moe_ffn_workspace_size(64, 8, 256, 128, 2)
    assert ok > 0
    assert moe.moe_ffn_workspace_size(64, 8, 200, 128, 2) == 0      # D % 128
    assert moe.moe_ffn_workspace_size(64, 8, 256, 100, 2) == 0      # H % 128
    assert moe.moe_ffn_workspace_size(64, 0, 256, 128, 2) == 0      # E >= 1
    assert moe.moe_ffn_workspace_size(64, 2000, 256, 128, 2) == 0   # E <= 1024
    assert moe.moe_ffn_workspace_size(64, 8, 256, 128, 0) == 0      # k >= 1
    assert moe.moe_ffn_workspace_size(-1, 8, 256, 128, 2) == 0
    # the split pipeline holds the gathered rows and the activation
    big = moe.moe_ffn_workspace_size(4096, 128, 2048, 768, 8, moe.MOE_BF16, moe.MOE_SPLIT)
    P = 4096 * 8
    s_max = (P + 128 * 127 + 127) // 128 * 128
    assert big >= s_max * (2048 + 768) * 2


def test_forward_rejects_bad_arguments_on_host():
    L = moe.lib()
    A = 1 << 20  # a fake, 16-byte aligned address: never dereferenced
    ws = 10 ** 9
    call = lambda *a: L.moe_ffn_forward(*a)
    base = [A, None, A, None, A, None, A, A, A, 64, 8, 256, 128, 2, 0, 1, A, ws, None]
    a = list(base); a[0] = None
    assert call(*a) == 1                                   # null x
    a = list(base); a[0] = A + 2
    assert call(*a) == 3                                   # misaligned x
    a = list(base); a[11] = 200
    assert call(*a) == 1                                   # D % 128
    a = list(base); a[14] = 5
    assert call(*a) == 1                                   # bad dtype
    a = list(base); a[1] = A
    assert call(*a) == 1                                   # scales given for bf16
    a = list(base); a[9] = 0
    assert call(*a) == 0                                   # T == 0: no-op
    a = list(base); a[17] = 16
    assert call(*a) in (5, 7)                              # workspace too small (or no device here)
    # MXFP4 weights: scales required, split pipeline only, weights 32-byte aligned
    mx4 = list(base); mx4[14] = 2; mx4[15] = 1; mx4[1] = mx4[3] = mx4[5] = A
    a = list(mx4); a[3] = None
    assert call(*a) == 1                                   # missing weight scales
    a = list(mx4); a[15] = 0
    assert call(*a) == 2                                   # fused pipeline: unsupported
    a = list(mx4); a[2] = A + 16
    assert call(*a) == 3                                   # w1 16- but not 32-byte aligned
    assert moe.moe_ffn_workspace_size(64, 8, 256, 128, 2, moe.MOE_MXFP4W, moe.MOE_SPLIT) == \
        moe.moe_ffn_workspace_size(64, 8, 256, 128, 2, moe.MOE_MXFP8, moe.MOE_SPLIT)


def test_header_compiles_as_c_and_cpp():
    import subprocess
    for lang, std in (("c", "c99"), ("c++", "c++17")):
        subprocess.run(["gcc", "-x", lang, f"-std={std}", "-Wall", "-Werror", "-fsyntax-only", HEADER], check=True)


def test_noalloc_route_size_limits_on_host():
    """The allocation-free routing call accepts problems up to T*k = 131072 with
    E = 1024 (its scratch layout fits the fixed array) and rejects larger ones
    before touching the device.  Without a GPU an accepted call stops at the
    device lookup (MOE_ERR_CUDA); a rejected one returns
    MOE_ERR_WORKSPACE_TOO_SMALL."""
    import torch
    L = moe.lib()
    A = 1 << 20
    if torch.cuda.is_available():
        pytest.skip("host-only check")
    assert L.moe_ffn_route_noalloc(A, A, 131072, 1024, 1, A, A, A, None, None) == 7
    assert L.moe_ffn_route_noalloc(A, A, 16384, 1024, 8, A, A, A, None, None) == 7
    assert L.moe_ffn_route_noalloc(A, A, 16385, 1024, 8, A, A, A, None, None) == 5


def test_extras_and_router_reject_bad_arguments_on_host():
    L = moe.lib()
    A = 1 << 20  # a fake, 16-byte aligned address: never dereferenced
    ws = 10 ** 9
    base = [A, None, A, None, A, None, A, A, A, 64, 8, 256, 128, 2, 0, 1]
    for limit, ns in ((-1.0, 0), (float("nan"), 0), (0.0, -1), (0.0, 1017)):
        ex = moe.MoeFFNExtras(limit, ns, None)
        assert L.moe_ffn_forward_ex(*base, ctypes.byref(ex), A, ws, None) == 1
    ex = moe.MoeFFNExtras(0.0, 0, A)                        # router logits with k > E
    b2 = list(base); b2[13] = 9
    assert L.moe_ffn_forward_ex(*b2, ctypes.byref(ex), A, ws, None) == 1
    assert L.moe_ffn_router_topk(A, 16, 8, 9, A, A, None) == 1     # k > E
    assert L.moe_ffn_router_topk(A, 16, 8, 0, A, A, None) == 1     # k < 1
    assert L.moe_ffn_router_topk(A + 2, 16, 8, 2, A, A, None) == 3  # misaligned logits
    assert L.moe_ffn_router_topk(A, 0, 8, 2, A, A, None) == 0      # T == 0: no-op
    assert moe.moe_ffn_workspace_size_ex(64, 8, 256, 128, 2, 0) == moe.moe_ffn_workspace_size(64, 8, 256, 128, 2)
    assert moe.moe_ffn_workspace_size_ex(64, 8, 256, 128, 2, 2) > moe.moe_ffn_workspace_size(64, 10, 256, 128, 4)
    assert moe.moe_ffn_workspace_size_ex(64, 1020, 256, 128, 2, 5) == 0  # E + n_shared > 1024


def test_widen_mxfp4_rejects_bad_arguments_on_host():
    L = moe.lib()
    A = 1 << 20  # a fake, 16-byte aligned address: never dereferenced
    assert L.moe_ffn_widen_mxfp4_weights(A, 48, A, None) == 1        # not a multiple of 32
    assert L.moe_ffn_widen_mxfp4_weights(A, -32, A, None) == 1
    assert L.moe_ffn_widen_mxfp4_weights(None, 64, A, None) == 1
    assert L.moe_ffn_widen_mxfp4_weights(A + 8, 64, A, None) == 3     # misaligned input
    assert L.moe_ffn_widen_mxfp4_weights(A, 64, A + 4, None) == 3     # misaligned output
    assert L.moe_ffn_widen_mxfp4_weights(None, 0, None, None) == 0    # nothing to do


def test_binding_refuses_host_and_strided_tensors():
    import torch
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        moe._p(x)
    with pytest.raises(ValueError):
        moe._p(x.t())
    assert moe._p(None) is None and moe._p(1 << 20) == 1 << 20
    with pytest.raises(ValueError, match="CUDA"):
        moe.moe_ffn_router_topk(torch.zeros(4, 8), 2, torch.zeros(4, 2, dtype=torch.int32), torch.zeros(4, 2))


def test_binding_checks_buffer_sizes():
    # sizes are checked before any pointer is taken, so CPU tensors show it here
    import torch
    T, E, D, H, k = 4, 2, 256, 128, 2
    x = torch.zeros(T, D, dtype=torch.bfloat16)
    w1 = torch.zeros(E, 2 * H, D, dtype=torch.bfloat16)
    w2 = torch.zeros(E, D, H - 1, dtype=torch.bfloat16)            # one column short
    ids = torch.zeros(T, k, dtype=torch.int32)
    tw = torch.zeros(T, k)
    out = torch.zeros(T, D, dtype=torch.bfloat16)
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    with pytest.raises(ValueError, match="w2"):
        moe.moe_ffn_forward(x, w1, w2, ids, tw, out, E=E, D=D, H=H, k=k, workspace=ws)
    with pytest.raises(ValueError, match="slot_of_pair"):
        moe.moe_ffn_route(ids, tw, T, E, k, torch.zeros(E, dtype=torch.int32), torch.zeros(E + 1, dtype=torch.int32),
                          torch.zeros(T * k - 1, dtype=torch.int32), ws)
    with pytest.raises(ValueError, match="logits"):
        moe.moe_ffn_router_topk(torch.zeros(T, E - 1), k, ids, tw, E=E)


def test_binding_leaves_out_of_range_shared_counts_to_the_c_abi():
    import torch
    T, E, D, H, k = 4, 4, 256, 128, 2
    t = lambda *s, dt=torch.bfloat16: torch.zeros(*s, dtype=dt)
    args = (t(T, D), t(E, 2 * H, D), t(E, D, H), t(T, k, dt=torch.int32), t(T, k, dt=torch.float32), t(T, D))
    # the size check must not turn an invalid count into a size error (the host
    # tensors then fail the device check, after the size check passed)
    for ns in (-1, 1021):
        with pytest.raises(ValueError, match="CUDA"):
            moe.moe_ffn_forward_ex(*args, E=E, D=D, H=H, k=k, workspace=t(1 << 20, dt=torch.uint8), n_shared=ns)


def test_route_padded_capacity_and_host_checks():
    def s_max(T, E, k):
        P = T * k
        return max(128, (P + min(E, P) * 127 + 127) // 128 * 128)
    for T, E, k in ((4096, 128, 8), (3, 1024, 4), (64, 8, 2), (1, 1, 1), (131072, 128, 8)):
        assert moe.moe_ffn_route_padded_slots(T, E, k) == s_max(T, E, k)
    assert moe.moe_ffn_route_padded_slots(4, 0, 2) == 0
    assert moe.moe_ffn_route_padded_slots(-1, 8, 2) == 0
    L = moe.lib()
    ws = ctypes.create_string_buffer(1 << 16)
    nul = [None] * 6
    # T = 0, null arrays and a missing workspace are refused before any launch
    assert L.moe_ffn_route_padded(None, None, 0, 8, 2, *nul, ctypes.addressof(ws), 1 << 16, None) == 1
    assert L.moe_ffn_route_padded(None, None, 4, 8, 2, *nul, ctypes.addressof(ws), 1 << 16, None) == 1
    assert L.moe_ffn_route_padded(1, 1, 4, 8, 2, 1, 1, 1, 1, 1, 1, None, 0, None) == 1


def test_workspace_holds_fp32_row_sums_for_large_k():
    # from k = 9 on the split pipeline sums each token's rows in an fp32 [T, D] accumulator
    T, E, D, H = 1000, 64, 512, 256
    for dtype in (moe.MOE_BF16, moe.MOE_MXFP8):
        k8 = moe.moe_ffn_workspace_size(T, E, D, H, 8, dtype, moe.MOE_SPLIT)
        k9 = moe.moe_ffn_workspace_size(T, E, D, H, 9, dtype, moe.MOE_SPLIT)
        assert k9 >= k8 + T * D * 4


def test_host_entry_sizes_and_rejects_bad_arguments_on_host():
    one = moe.moe_ffn_workspace_size(300, 16, 512, 256, 4)
    h = moe.moe_ffn_host_workspace_size(300, 16, 512, 256, 4)
    # the forward workspace of a chunk plus two sets of staging buffers
    assert h >= one + 2 * (300 * 512 * 2 + 2 * 300 * 4 * 4 + 300 * 512 * 2)
    assert moe.moe_ffn_host_workspace_size(300, 16, 512, 256, 4, chunk_tokens=64) < h
    # automatic chunks: whole problems up to 8192 tokens, else T / 8 within [4096, 16384]
    size = lambda T, c=0: moe.moe_ffn_host_workspace_size(T, 16, 512, 256, 4, chunk_tokens=c)
    assert size(200000) == size(16384, 16384)
    assert size(16384) == size(16384, 4096)
    assert size(50000) == size(50000, 6272)
    assert size(8192) == size(8192, 8192)
    assert moe.moe_ffn_host_workspace_size(300, 16, 512, 256, 4, dtype=moe.MOE_NVFP4) == 0
    assert moe.moe_ffn_host_workspace_size(300, 16, 512, 256, 4, chunk_tokens=-1) == 0
    L = moe.lib()
    A = 1 << 20  # fake addresses: never dereferenced
    base = [A, None, A, None, A, None, A, A, A, 300, 16, 512, 256, 4, 0, 1, 0, A, 10 ** 9, None]
    a = list(base); a[0] = None
    assert L.moe_ffn_forward_host(*a) == 1                  # null x
    a = list(base); a[8] = None
    assert L.moe_ffn_forward_host(*a) == 1                  # null out
    a = list(base); a[16] = -5
    assert L.moe_ffn_forward_host(*a) == 1                  # negative chunk size
    a = list(base); a[14] = 3
    assert L.moe_ffn_forward_host(*a) == 1                  # NVFP4 has its own entry point
    a = list(base); a[14] = 1
    assert L.moe_ffn_forward_host(*a) == 1                  # MXFP8 without x scales
    a = list(base); a[9] = 0
    assert L.moe_ffn_forward_host(*a) == 0                  # T == 0: no-op
    a = list(base); a[18] = 1024
    assert L.moe_ffn_forward_host(*a) == 5                  # workspace too small


def test_option_values_are_checked_on_host():
    # each option takes its documented values; anything else is refused and
    # leaves the option as it was
    cases = {
        moe.MOE_OPT_DOWN_EPI8: ([0, 1], [2, -1]),
        moe.MOE_OPT_MX_PAIRS: ([0, 1, 2], [3]),
        moe.MOE_OPT_UP_SWAP: ([0, 1], [2]),
        moe.MOE_OPT_ROUTE_TPB: ([0, 64, 128, 256], [32, 100, 512]),
        moe.MOE_OPT_MX_SWAP: ([0, 1, 2], [3]),
        moe.MOE_OPT_HOST_RAMP: ([0, 1], [2]),
    }
    defaults = {moe.MOE_OPT_DOWN_EPI8: 1, moe.MOE_OPT_MX_PAIRS: 0, moe.MOE_OPT_UP_SWAP: 1,
                moe.MOE_OPT_ROUTE_TPB: 0, moe.MOE_OPT_MX_SWAP: 0, moe.MOE_OPT_HOST_RAMP: 1}
    try:
        for opt, (good, bad) in cases.items():
            for v in good:
                assert moe.moe_ffn_set_option(opt, v) == 0, (opt, v)
            for v in bad:
                assert moe.lib().moe_ffn_set_option(opt, v) == 1, (opt, v)
        assert moe.lib().moe_ffn_set_option(999, 0) == 1          # unknown option
    finally:
        for opt, v in defaults.items():
            moe.moe_ffn_set_option(opt, v)


def test_routing_block_size_option_sizes_the_workspace():
    # fewer tokens per routing block -> more blocks -> a larger per-block count table
    base = moe.moe_ffn_workspace_size(4096, 128, 2048, 768, 8)
    moe.moe_ffn_set_option(moe.MOE_OPT_ROUTE_TPB, 64)
    try:
        small_blocks = moe.moe_ffn_workspace_size(4096, 128, 2048, 768, 8)
    finally:
        moe.moe_ffn_set_option(moe.MOE_OPT_ROUTE_TPB, 0)
    assert small_blocks >= base + (4096 // 64 - 4096 // 256) * 128 * 4 - 256


def test_host_entry_binding_checks_its_host_tensors():
    # sizes and the host side are checked before any pointer reaches the C ABI
    import torch
    T, E, D, H, k = 4, 2, 256, 128, 2
    x = torch.zeros(T, D, dtype=torch.bfloat16)
    w1 = torch.zeros(E, 2 * H, D, dtype=torch.bfloat16)
    w2 = torch.zeros(E, D, H, dtype=torch.bfloat16)
    ids = torch.zeros(T, k, dtype=torch.int32)
    tw = torch.zeros(T, k)
    out = torch.zeros(T, D, dtype=torch.bfloat16)
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    A = 1 << 20  # device weights as raw addresses (no GPU here); never reached: a host check fails first
    call = lambda **kw: moe.moe_ffn_forward_host(kw.get("x", x), A, A, kw.get("ids", ids), kw.get("tw", tw),
                                                 kw.get("out", out), E=E, D=D, H=H, k=k, workspace=A)
    with pytest.raises(ValueError, match="out"):
        call(out=torch.zeros(T, D - 1, dtype=torch.bfloat16))      # short output
    with pytest.raises(ValueError, match="topk_ids"):
        call(ids=torch.zeros(T, k - 1, dtype=torch.int32))
    with pytest.raises(ValueError, match="contiguous"):
        call(x=torch.zeros(D, T, dtype=torch.bfloat16).t())
    with pytest.raises(ValueError, match="T is required"):
        call(x=1 << 20)                                             # a raw address carries no shape
    with pytest.raises(ValueError, match="w2"):                     # weight sizes are checked like moe_ffn_forward's
        moe.moe_ffn_forward_host(x, w1, torch.zeros(E, D, H - 1, dtype=torch.bfloat16), ids, tw, out,
                                 E=E, D=D, H=H, k=k, workspace=ws)
