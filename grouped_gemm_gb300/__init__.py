"""Python binding of the GB300 MoE SwiGLU FFN library (libmoe_ffn.so).

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels behind the C ABI declared in ``include/moe_ffn.h``.  The function names
are the C names.  Tensors are torch tensors (device memory and streams come
from PyTorch); their data pointers are passed through unchanged.  There is no
CPU fallback: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "MOE_BF16", "MOE_MXFP8", "MOE_MXFP4W", "MOE_NVFP4", "MOE_FUSED", "MOE_SPLIT", "MoeFFNError", "library_path", "lib",
    "moe_ffn_workspace_size", "moe_ffn_workspace_init", "moe_ffn_forward", "moe_ffn_forward_logits", "moe_ffn_forward_ex", "MoeFFNExtras",
    "moe_ffn_host_workspace_size", "moe_ffn_forward_host",
    "moe_ffn_workspace_size_ex", "moe_ffn_router_topk", "moe_ffn_route", "moe_ffn_route_noalloc",
    "moe_ffn_sync_status", "moe_ffn_set_wait_limit_ns", "moe_ffn_profile_enable", "moe_ffn_profile_read", "moe_ffn_profile_stage_kernel", "moe_ffn_set_option", "MOE_OPT_GATHER", "moe_ffn_prepare_mxfp8_weights", "moe_ffn_widen_mxfp4_weights", "moe_ffn_debug_mx_quantize", "moe_ffn_status_string", "alloc_workspace",
]

MOE_BF16, MOE_MXFP8, MOE_MXFP4W, MOE_NVFP4 = 0, 1, 2, 3
MOE_FUSED, MOE_SPLIT = 0, 1
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_MISALIGNED",
                4: "MOE_ERR_BAD_ROUTING", 5: "MOE_ERR_WORKSPACE_TOO_SMALL", 6: "MOE_ERR_DEVICE_TIMEOUT",
                7: "MOE_ERR_CUDA"}

_lock = threading.Lock()
_lib = None


class MoeFFNExtras(ctypes.Structure):
    """moe_ffn_extras_t: clamped SwiGLU limit, shared experts, router logits."""
    _fields_ = [("swiglu_limit", ctypes.c_float), ("n_shared", ctypes.c_int), ("router_logits", ctypes.c_void_p)]


class NvFp4Scales(ctypes.Structure):
    """moe_ffn_nvfp4_scales_t: device pointers to the fp32 global scales."""
    _fields_ = [("x_gs", ctypes.c_void_p), ("w1_gs", ctypes.c_void_p), ("w2_gs", ctypes.c_void_p),
                ("act_gs", ctypes.c_void_p)]


class MoeFFNError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({moe_ffn_status_string(status)})")


def library_path() -> str:
    from . import build as _build
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libmoe_ffn.so, building it first if the sources are newer."""
    global _lib
    with _lock:
        if _lib is None:
            from . import build as _build
            path = _build.build()
            L = ctypes.CDLL(path)
            c = ctypes
            vp, i, sz = c.c_void_p, c.c_int, c.c_size_t
            L.moe_ffn_workspace_size.argtypes = [i, i, i, i, i, i, i]
            L.moe_ffn_workspace_size.restype = sz
            L.moe_ffn_workspace_init.argtypes = [vp, sz, vp]
            L.moe_ffn_workspace_init.restype = i
            L.moe_ffn_forward.argtypes = [vp] * 9 + [i] * 7 + [vp, sz, vp]
            L.moe_ffn_forward.restype = i
            L.moe_ffn_router_topk.argtypes = [vp, i, i, i, vp, vp, vp]
            L.moe_ffn_router_topk.restype = i
            L.moe_ffn_forward_logits.argtypes = [vp] * 10 + [i] * 7 + [vp, sz, vp]
            L.moe_ffn_forward_logits.restype = i
            L.moe_ffn_host_workspace_size.argtypes = [i] * 8
            L.moe_ffn_host_workspace_size.restype = sz
            L.moe_ffn_forward_host.argtypes = [vp] * 9 + [i] * 8 + [vp, sz, vp]
            L.moe_ffn_forward_host.restype = i
            L.moe_ffn_workspace_size_ex.argtypes = [i] * 8
            L.moe_ffn_workspace_size_ex.restype = sz
            L.moe_ffn_forward_ex.argtypes = [vp] * 9 + [i] * 7 + [c.POINTER(MoeFFNExtras), vp, sz, vp]
            L.moe_ffn_forward_ex.restype = i
            L.moe_ffn_route.argtypes = [vp, vp, i, i, i, vp, vp, vp, vp, sz, vp]
            L.moe_ffn_route.restype = i
            L.moe_ffn_route_noalloc.argtypes = [vp, vp, i, i, i, vp, vp, vp, vp, vp]
            L.moe_ffn_route_noalloc.restype = i
            L.moe_ffn_route_padded_slots.argtypes = [i, i, i]
            L.moe_ffn_route_padded_slots.restype = c.c_int64
            L.moe_ffn_route_padded.argtypes = [vp, vp, i, i, i, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            L.moe_ffn_route_padded.restype = i
            L.moe_ffn_prepare_mxfp8_weights.argtypes = [vp, vp, vp, vp, i, i, i, vp]
            L.moe_ffn_prepare_mxfp8_weights.restype = i
            L.moe_ffn_prepare_nvfp4_weights.argtypes = [vp, vp, vp, vp, i, i, i, vp]
            L.moe_ffn_prepare_nvfp4_weights.restype = i
            L.moe_ffn_forward_nvfp4.argtypes = [vp] * 6 + [c.POINTER(NvFp4Scales)] + [vp] * 3 + [i] * 5 + [vp, sz, vp]
            L.moe_ffn_forward_nvfp4.restype = i
            L.moe_ffn_widen_mxfp4_weights.argtypes = [vp, c.c_int64, vp, vp]
            L.moe_ffn_widen_mxfp4_weights.restype = i
            L.moe_ffn_debug_mx_quantize.argtypes = [vp, c.c_int64, vp, vp, vp]
            L.moe_ffn_debug_mx_quantize.restype = i
            L.moe_ffn_sync_status.argtypes = [vp, vp]
            L.moe_ffn_sync_status.restype = i
            L.moe_ffn_set_wait_limit_ns.argtypes = [c.c_uint64]
            L.moe_ffn_set_wait_limit_ns.restype = None
            L.moe_ffn_set_option.argtypes = [i, c.c_longlong]
            L.moe_ffn_set_option.restype = i
            L.moe_ffn_profile_enable.argtypes = [i]
            L.moe_ffn_profile_enable.restype = i
            L.moe_ffn_profile_read.argtypes = [c.POINTER(c.c_float), i, c.POINTER(c.c_int)]
            L.moe_ffn_profile_read.restype = i
            L.moe_ffn_profile_stage_kernel.argtypes = [i]
            L.moe_ffn_profile_stage_kernel.restype = c.c_char_p
            L.moe_ffn_status_string.argtypes = [i]
            L.moe_ffn_status_string.restype = c.c_char_p
            _lib = L
    return _lib


def _p(t):
    """Device pointer of a tensor, None for None, ints pass through.  Every
    array argument of the C ABI is a dense device array, so a tensor must be
    a contiguous CUDA tensor: anything else is refused here rather than
    handed to a kernel."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"expected a contiguous tensor, got strides {tuple(t.stride())}")
    return t.data_ptr()


def _need(t, nbytes, name):
    """A tensor argument must hold at least nbytes (the kernels read and write
    exactly the extents the sizes imply; a raw int pointer is the caller's
    responsibility)."""
    if t is None or isinstance(t, int):
        return
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name} holds {have} bytes, the call needs {int(nbytes)}")


def _need_forward(x, x_sf, w1, w1_sf, w2, w2_sf, topk_ids, topk_w, out, T, E, D, H, k, dtype):
    eb = 2 if dtype == MOE_BF16 else 1
    wb = 0.5 if dtype == MOE_MXFP4W else eb    # packed E2M1 weights: two codes per byte
    _need(x, T * D * eb, "x")
    _need(w1, E * 2 * H * D * wb, "w1")
    _need(w2, E * D * H * wb, "w2")
    _need(out, T * D * 2, "out")
    _need(topk_ids, T * k * 4, "topk_ids")
    _need(topk_w, T * k * 4, "topk_w")
    if dtype != MOE_BF16:
        _need(x_sf, T * D // 32, "x_sf")
        _need(w1_sf, E * 2 * H * D // 32, "w1_sf")
        _need(w2_sf, E * D * H // 32, "w2_sf")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> int:
    if status != 0:
        raise MoeFFNError(status, where)
    return status


def moe_ffn_status_string(status: int) -> str:
    return lib().moe_ffn_status_string(int(status)).decode()


def moe_ffn_workspace_size(T, E, D, H, k, dtype=MOE_BF16, pipeline=MOE_SPLIT) -> int:
    return int(lib().moe_ffn_workspace_size(T, E, D, H, k, dtype, pipeline))


def moe_ffn_workspace_init(workspace, stream=None) -> int:
    return _check(lib().moe_ffn_workspace_init(_p(workspace), workspace.numel() * workspace.element_size(),
                                               _stream(stream)), "moe_ffn_workspace_init")


def moe_ffn_workspace_size_ex(T, E, D, H, k, n_shared, dtype=MOE_BF16, pipeline=MOE_SPLIT) -> int:
    return lib().moe_ffn_workspace_size_ex(T, E, D, H, k, n_shared, dtype, pipeline)


def alloc_workspace(T, E, D, H, k, dtype=MOE_BF16, pipeline=MOE_SPLIT, device="cuda", n_shared=0):
    """A caller-owned workspace tensor of the right size, status words zeroed
    (sized for moe_ffn_forward_ex with n_shared shared experts)."""
    import torch
    n = moe_ffn_workspace_size_ex(T, E, D, H, k, n_shared, dtype, pipeline)
    if n == 0:
        raise MoeFFNError(1, "moe_ffn_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_ffn_workspace_init(ws)
    return ws


def moe_ffn_forward(x, w1, w2, topk_ids, topk_w, out, *, E, D, H, k, workspace, dtype=MOE_BF16,
                    pipeline=MOE_SPLIT, x_sf=None, w1_sf=None, w2_sf=None, T=None, stream=None,
                    check=True) -> int:
    T = x.shape[0] if T is None else T
    _need_forward(x, x_sf, w1, w1_sf, w2, w2_sf, topk_ids, topk_w, out, T, E, D, H, k, dtype)
    st = lib().moe_ffn_forward(_p(x), _p(x_sf), _p(w1), _p(w1_sf), _p(w2), _p(w2_sf), _p(topk_ids), _p(topk_w),
                               _p(out), T, E, D, H, k, dtype, pipeline, _p(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    return _check(st, "moe_ffn_forward") if check else st


def moe_ffn_host_workspace_size(T, E, D, H, k, dtype=MOE_BF16, pipeline=MOE_SPLIT, chunk_tokens=0) -> int:
    return int(lib().moe_ffn_host_workspace_size(T, chunk_tokens, E, D, H, k, dtype, pipeline))


def _host_p(t, nbytes, name):
    """Address of a host (CPU) tensor argument holding at least nbytes (a raw
    int address is passed through: its extent is the caller's responsibility)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if t.is_cuda:
        raise ValueError(f"{name}: expected a host tensor, got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    _need(t, nbytes, name)
    return t.data_ptr()


def moe_ffn_forward_host(x, w1, w2, topk_ids, topk_w, out, *, E, D, H, k, workspace, dtype=MOE_BF16,
                         pipeline=MOE_SPLIT, x_sf=None, w1_sf=None, w2_sf=None, chunk_tokens=0, T=None, stream=None,
                         check=True) -> int:
    """moe_ffn_forward_host: x (x_sf), topk_ids, topk_w and out are host tensors
    (page-locked for overlapped copies), the weights and workspace CUDA tensors."""
    if T is None:
        if isinstance(x, int):
            raise ValueError("T is required when x is a raw address")
        T = x.shape[0]
    eb = 2 if dtype == MOE_BF16 else 1
    _need_forward(None, None, w1, w1_sf, w2, w2_sf, None, None, None, T, E, D, H, k, dtype)
    st = lib().moe_ffn_forward_host(
        _host_p(x, T * D * eb, "x"), _host_p(x_sf, T * D // 32, "x_sf"), _p(w1), _p(w1_sf), _p(w2), _p(w2_sf),
        _host_p(topk_ids, T * k * 4, "topk_ids"), _host_p(topk_w, T * k * 4, "topk_w"),
        _host_p(out, T * D * 2, "out"), T, E, D, H, k, dtype, pipeline, chunk_tokens, _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    return _check(st, "moe_ffn_forward_host") if check else st


def moe_ffn_forward_logits(x, w1, w2, router_logits, topk_ids, topk_w, out, *, E, D, H, k, workspace,
                           dtype=MOE_BF16, pipeline=MOE_SPLIT, x_sf=None, w1_sf=None, w2_sf=None, T=None,
                           stream=None, check=True) -> int:
    """moe_ffn_forward from router logits [T, E] fp32; topk_ids / topk_w [T, k]
    are written by the call."""
    T = x.shape[0] if T is None else T
    _need_forward(x, x_sf, w1, w1_sf, w2, w2_sf, topk_ids, topk_w, out, T, E, D, H, k, dtype)
    _need(router_logits, T * E * 4, "router_logits")
    st = lib().moe_ffn_forward_logits(_p(x), _p(x_sf), _p(w1), _p(w1_sf), _p(w2), _p(w2_sf), _p(router_logits),
                                      _p(topk_ids), _p(topk_w), _p(out), T, E, D, H, k, dtype, pipeline,
                                      _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    return _check(st, "moe_ffn_forward_logits") if check else st


def moe_ffn_forward_ex(x, w1, w2, topk_ids, topk_w, out, *, E, D, H, k, workspace, dtype=MOE_BF16,
                       pipeline=MOE_SPLIT, x_sf=None, w1_sf=None, w2_sf=None, T=None, swiglu_limit=0.0, n_shared=0,
                       router_logits=None, stream=None, check=True) -> int:
    """moe_ffn_forward with a clamped SwiGLU (swiglu_limit > 0), n_shared shared
    experts stored after the E routed ones, and/or router logits [T, E]."""
    T = x.shape[0] if T is None else T
    ns = int(n_shared)
    ns = ns if 0 <= ns <= 1024 - E else 0   # an out-of-range count is the C ABI's to reject
    _need_forward(x, x_sf, w1, w1_sf, w2, w2_sf, topk_ids, topk_w, out, T, E + ns, D, H, k, dtype)
    _need(router_logits, T * E * 4, "router_logits")
    ex = MoeFFNExtras(float(swiglu_limit), int(n_shared), _p(router_logits))
    st = lib().moe_ffn_forward_ex(_p(x), _p(x_sf), _p(w1), _p(w1_sf), _p(w2), _p(w2_sf), _p(topk_ids), _p(topk_w),
                                  _p(out), T, E, D, H, k, dtype, pipeline, ctypes.byref(ex), _p(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    return _check(st, "moe_ffn_forward_ex") if check else st


def moe_ffn_router_topk(logits, k, topk_ids, topk_w, T=None, E=None, stream=None, check=True) -> int:
    """Top-k experts and softmax-renormalized weights of router logits [T, E]."""
    T = logits.shape[0] if T is None else T
    E = logits.shape[1] if E is None else E
    _need(logits, T * E * 4, "logits")
    _need(topk_ids, T * k * 4, "topk_ids")
    _need(topk_w, T * k * 4, "topk_w")
    st = lib().moe_ffn_router_topk(_p(logits), T, E, k, _p(topk_ids), _p(topk_w), _stream(stream))
    return _check(st, "moe_ffn_router_topk") if check else st


def _need_route(topk_ids, topk_w, T, E, k, counts, offsets, slot_of_pair):
    _need(topk_ids, T * k * 4, "topk_ids")
    _need(topk_w, T * k * 4, "topk_w")
    _need(counts, E * 4, "counts")
    _need(offsets, (E + 1) * 4, "offsets")
    _need(slot_of_pair, T * k * 4, "slot_of_pair")


def moe_ffn_route(topk_ids, topk_w, T, E, k, counts, offsets, slot_of_pair, workspace, stream=None,
                  check=True) -> int:
    _need_route(topk_ids, topk_w, T, E, k, counts, offsets, slot_of_pair)
    st = lib().moe_ffn_route(_p(topk_ids), _p(topk_w), T, E, k, _p(counts), _p(offsets), _p(slot_of_pair),
                             _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    return _check(st, "moe_ffn_route") if check else st


def moe_ffn_route_padded_slots(T, E, k) -> int:
    """Capacity S_max of the padded routing tables (0 for an invalid shape)."""
    return int(lib().moe_ffn_route_padded_slots(T, E, k))


def moe_ffn_route_padded(topk_ids, topk_w, T, E, k, pad_offsets, expert_of_rb, pair_info, row_tok, slot_w, n_blocks,
                         workspace, stream=None, check=True) -> int:
    """The padded routing tables the grouped GEMMs consume (pad_offsets [E+1],
    expert_of_rb and pair_info [S_max/128], row_tok and slot_w [S_max],
    n_blocks [2] = row blocks and pairs), S_max = moe_ffn_route_padded_slots."""
    smax = moe_ffn_route_padded_slots(T, E, k)
    _need(topk_ids, T * k * 4, "topk_ids")
    _need(topk_w, T * k * 4, "topk_w")
    _need(pad_offsets, (E + 1) * 4, "pad_offsets")
    _need(expert_of_rb, smax // 128 * 4, "expert_of_rb")
    _need(pair_info, smax // 128 * 4, "pair_info")
    _need(row_tok, smax * 4, "row_tok")
    _need(slot_w, smax * 4, "slot_w")
    _need(n_blocks, 8, "n_blocks")
    st = lib().moe_ffn_route_padded(_p(topk_ids), _p(topk_w), T, E, k, _p(pad_offsets), _p(expert_of_rb),
                                    _p(pair_info), _p(row_tok), _p(slot_w), _p(n_blocks), _p(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    return _check(st, "moe_ffn_route_padded") if check else st


def moe_ffn_route_noalloc(topk_ids, topk_w, T, E, k, counts, offsets, slot_of_pair, status_bits=None, stream=None,
                          check=True) -> int:
    """Routing permutation without a caller workspace, for callers that
    cannot allocate device memory (scratch is a fixed array inside the
    library; T*k <= 131072).  Calls on one device must not overlap."""
    _need_route(topk_ids, topk_w, T, E, k, counts, offsets, slot_of_pair)
    _need(status_bits, 4, "status_bits")
    st = lib().moe_ffn_route_noalloc(_p(topk_ids), _p(topk_w), T, E, k, _p(counts), _p(offsets),
                                     _p(slot_of_pair), _p(status_bits), _stream(stream))
    return _check(st, "moe_ffn_route_noalloc") if check else st


def moe_ffn_prepare_mxfp8_weights(w1_sf, w2_sf, w1_sf_packed, w2_sf_packed, E, D, H, stream=None) -> int:
    for t, n, name in ((w1_sf, E * 2 * H * D // 32, "w1_sf"), (w1_sf_packed, E * 2 * H * D // 32, "w1_sf_packed"),
                       (w2_sf, E * D * H // 32, "w2_sf"), (w2_sf_packed, E * D * H // 32, "w2_sf_packed")):
        _need(t, n, name)
    return _check(lib().moe_ffn_prepare_mxfp8_weights(_p(w1_sf), _p(w2_sf), _p(w1_sf_packed), _p(w2_sf_packed), E, D,
                                                       H, _stream(stream)), "moe_ffn_prepare_mxfp8_weights")


def moe_ffn_prepare_nvfp4_weights(w1_sf, w2_sf, w1_sf_packed, w2_sf_packed, E, D, H, stream=None) -> int:
    """Repack NVFP4 weight scales (e4m3 bytes, one per 16 elements) into the
    kernels' 512-byte tiles."""
    for t, n, name in ((w1_sf, E * 2 * H * D // 16, "w1_sf"), (w1_sf_packed, E * 2 * H * D // 16, "w1_sf_packed"),
                       (w2_sf, E * D * H // 16, "w2_sf"), (w2_sf_packed, E * D * H // 16, "w2_sf_packed")):
        _need(t, n, name)
    return _check(lib().moe_ffn_prepare_nvfp4_weights(_p(w1_sf), _p(w2_sf), _p(w1_sf_packed), _p(w2_sf_packed), E, D,
                                                       H, _stream(stream)), "moe_ffn_prepare_nvfp4_weights")


def moe_ffn_forward_nvfp4(x, x_sf, w1, w1_sf, w2, w2_sf, x_gs, w1_gs, w2_gs, act_gs, topk_ids, topk_w, out, *, E, D,
                          H, k, workspace, T=None, stream=None, check=True) -> int:
    """Forward pass with NVFP4 operands (split pipeline): packed E2M1 codes
    (uint8), e4m3 scales per 16 (x_sf row-major, w*_sf repacked), fp32 global
    scales as device tensors x_gs [1], w1_gs [E], w2_gs [E], act_gs [1]."""
    T = x.shape[0] if T is None else T
    for t, n, name in ((x, T * D // 2, "x"), (x_sf, T * D // 16, "x_sf"), (w1, E * 2 * H * D // 2, "w1"),
                       (w1_sf, E * 2 * H * D // 16, "w1_sf"), (w2, E * D * H // 2, "w2"),
                       (w2_sf, E * D * H // 16, "w2_sf"), (x_gs, 4, "x_gs"), (w1_gs, 4 * E, "w1_gs"),
                       (w2_gs, 4 * E, "w2_gs"), (act_gs, 4, "act_gs"), (topk_ids, T * k * 4, "topk_ids"),
                       (topk_w, T * k * 4, "topk_w"), (out, T * D * 2, "out")):
        _need(t, n, name)
    gs = NvFp4Scales(_p(x_gs), _p(w1_gs), _p(w2_gs), _p(act_gs))
    st = lib().moe_ffn_forward_nvfp4(_p(x), _p(x_sf), _p(w1), _p(w1_sf), _p(w2), _p(w2_sf), ctypes.byref(gs),
                                     _p(topk_ids), _p(topk_w), _p(out), T, E, D, H, k, _p(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream))
    return _check(st, "moe_ffn_forward_nvfp4") if check else st


def moe_ffn_widen_mxfp4_weights(w_fp4, w_e4m3, stream=None) -> int:
    """MXFP4 weight codes (uint8, two per byte) -> e4m3 codes (uint8, one per byte)."""
    if w_fp4.numel() * 2 != w_e4m3.numel():
        raise ValueError(f"w_fp4 holds {w_fp4.numel() * 2} codes, w_e4m3 {w_e4m3.numel()}")
    return _check(lib().moe_ffn_widen_mxfp4_weights(_p(w_fp4), w_e4m3.numel(), _p(w_e4m3), _stream(stream)),
                  "moe_ffn_widen_mxfp4_weights")


def moe_ffn_debug_mx_quantize(x, q, sf, stream=None) -> int:
    _need(q, x.numel(), "q")
    _need(sf, x.numel() // 32, "sf")
    return _check(lib().moe_ffn_debug_mx_quantize(_p(x), x.numel(), _p(q), _p(sf), _stream(stream)),
                  "moe_ffn_debug_mx_quantize")


def moe_ffn_sync_status(workspace, stream=None) -> int:
    """Synchronize and return (and clear) the device-side status: 0, 4 or 6."""
    return int(lib().moe_ffn_sync_status(_p(workspace), _stream(stream)))


MOE_OPT_GATHER = 0
MOE_OPT_L2_PREFETCH = 1
MOE_OPT_TEST_STALL = 2
MOE_OPT_UP_PAIRS = 3
MOE_OPT_DYNAMIC_TILES = 4
MOE_OPT_TILE_COLS = 5
MOE_OPT_SWAP_AB = 6
MOE_OPT_FUSED_CLUSTER = 7
MOE_OPT_PAIR_MMA = 8
MOE_OPT_PAIR_SWAP = 9
MOE_OPT_ROUTE_COOP = 10
MOE_OPT_OUT_L2_HINT = 11
MOE_OPT_GATHER_BLOCKS = 12
MOE_OPT_L2_POLICY = 13
MOE_OPT_ROUTER_FUSED = 14
MOE_OPT_PREFETCH_MB = 15
MOE_OPT_WIDE_UP = 16
MOE_OPT_TILE_M = 17
MOE_OPT_FUSED_DSMEM = 18
MOE_OPT_HALF_PAIR_M128 = 19
MOE_OPT_ROUTE_SMALL_PAIRS = 20
MOE_OPT_DOWN_BANDS = 21
MOE_OPT_DOWN_EPI8 = 22
MOE_OPT_MX_PAIRS = 23
MOE_OPT_UP_SWAP = 24
MOE_OPT_ROUTE_TPB = 25
MOE_OPT_MX_SWAP = 26
MOE_OPT_HOST_RAMP = 27


def moe_ffn_set_option(option: int, value: int) -> int:
    return _check(lib().moe_ffn_set_option(int(option), int(value)), "moe_ffn_set_option")


def moe_ffn_profile_enable(on: bool) -> int:
    return _check(lib().moe_ffn_profile_enable(1 if on else 0), "moe_ffn_profile_enable")


def moe_ffn_profile_read() -> list:
    """Stage durations (ms) of the most recent profiled forward call."""
    buf = (ctypes.c_float * 8)()
    n = ctypes.c_int(0)
    _check(lib().moe_ffn_profile_read(buf, 8, ctypes.byref(n)), "moe_ffn_profile_read")
    return [float(buf[i]) for i in range(n.value)]


def moe_ffn_profile_stage_kernel(stage: int):
    """Main kernel of one stage of the most recent profiled call (None if absent)."""
    r = lib().moe_ffn_profile_stage_kernel(int(stage))
    return None if r is None else r.decode()


def moe_ffn_set_wait_limit_ns(ns: int) -> None:
    lib().moe_ffn_set_wait_limit_ns(int(ns))
