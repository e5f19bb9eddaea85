"""CPU oracle for the routed MoE SwiGLU FFN forward pass (fp64).

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only the tests, ``__graft_entry__.smoke``
and the benchmark's cpu-baseline / reference legs may import this package.  It
shares nothing with the CUDA library; the arithmetic lives in ``oracle.c``
(plain C, compiled with gcc) and this module only marshals numpy arrays.

Page cited throughout: "Prime Flash MoE - Faster MoE Kernels optimized for
Blackwell" (sec. 1 "The computation", sec. 5 "The two epilogues", sec. 7 "The
MXFP8 variant"), and "Porting Block-Scaled GEMM Kernels from Blackwell to Rubin"
sec. 6.2 for the rounding of the MX scale.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

IN_BF16, IN_MXFP8, IN_MXFP4W = 0, 1, 2
ACT_EXACT, ACT_BF16, ACT_MXFP8, ACT_NVFP4 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc and OpenMP."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            c = ctypes
            lib.oracle_bf16_to_f64.argtypes = [c.c_uint16]
            lib.oracle_bf16_to_f64.restype = c.c_double
            lib.oracle_f32_to_bf16.argtypes = [c.c_float]
            lib.oracle_f32_to_bf16.restype = c.c_uint16
            lib.oracle_e4m3_to_f64.argtypes = [c.c_uint8]
            lib.oracle_e4m3_to_f64.restype = c.c_double
            lib.oracle_f64_to_e4m3.argtypes = [c.c_double]
            lib.oracle_f64_to_e4m3.restype = c.c_uint8
            lib.oracle_e8m0_to_f64.argtypes = [c.c_uint8]
            lib.oracle_e8m0_to_f64.restype = c.c_double
            lib.oracle_mx_scale_exponent.argtypes = [c.c_double]
            lib.oracle_mx_scale_exponent.restype = c.c_int
            lib.oracle_e2m1_to_f64.argtypes = [c.c_uint8]
            lib.oracle_e2m1_to_f64.restype = c.c_double
            lib.oracle_f64_to_e2m1.argtypes = [c.c_double]
            lib.oracle_f64_to_e2m1.restype = c.c_uint8
            lib.oracle_mx4_scale_exponent.argtypes = [c.c_double]
            lib.oracle_mx4_scale_exponent.restype = c.c_int
            lib.oracle_mx_quantize.argtypes = [c.c_void_p, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p]
            lib.oracle_mx_quantize.restype = None
            lib.oracle_route.argtypes = [c.c_int, c.c_int, c.c_int, c.c_void_p, c.c_int,
                                         c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p]
            lib.oracle_route.restype = c.c_int
            lib.oracle_router_topk.argtypes = [c.c_int, c.c_int, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p]
            lib.oracle_router_topk.restype = c.c_int
            lib.oracle_moe_ffn.argtypes = [c.c_int] * 6 + [c.c_void_p] * 8 + [c.c_int, c.c_void_p, c.c_int,
                                                                               c.c_void_p, c.c_int, c.c_double]
            lib.oracle_moe_ffn.restype = c.c_int
            vp, i_, d_ = c.c_void_p, c.c_int, c.c_double
            lib.oracle_nv4_quantize.argtypes = [vp, i_, d_, vp, vp, vp]
            lib.oracle_nv4_quantize.restype = None
            lib.oracle_moe_ffn_nvfp4.argtypes = ([i_] * 5 + [vp, vp, d_, vp, vp, vp, vp, vp, vp, vp, vp, i_, d_, vp, i_,
                                                              vp, i_, d_])
            lib.oracle_moe_ffn_nvfp4.restype = c.c_int
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = c.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- formats
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_bf16_to_f64(int(b)) for b in np.asarray(bits, np.uint16).ravel()]).reshape(
        np.shape(bits))


def f32_to_bf16(vals) -> np.ndarray:
    lib = _load()
    v = np.asarray(vals, np.float32)
    return np.array([lib.oracle_f32_to_bf16(float(x)) for x in v.ravel()], np.uint16).reshape(v.shape)


def e4m3_to_f64(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, np.uint8)
    return np.array([lib.oracle_e4m3_to_f64(int(q)) for q in c.ravel()]).reshape(c.shape)


def f64_to_e4m3(vals) -> np.ndarray:
    lib = _load()
    v = np.asarray(vals, np.float64)
    return np.array([lib.oracle_f64_to_e4m3(float(x)) for x in v.ravel()], np.uint8).reshape(v.shape)


def e2m1_to_f64(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, np.uint8)
    return np.array([lib.oracle_e2m1_to_f64(int(q)) for q in c.ravel()]).reshape(c.shape)


def f64_to_e2m1(vals) -> np.ndarray:
    lib = _load()
    v = np.asarray(vals, np.float64)
    return np.array([lib.oracle_f64_to_e2m1(float(x)) for x in v.ravel()], np.uint8).reshape(v.shape)


def mx4_scale_exponent(amax: float) -> int:
    return _load().oracle_mx4_scale_exponent(float(amax))


def mx_scale_exponent(amax: float) -> int:
    return _load().oracle_mx_scale_exponent(float(amax))


def mx_quantize(a: np.ndarray):
    """Per-32 MXFP8 quantization of a 1-D array; returns (codes, scale bytes, dequantized)."""
    a = np.ascontiguousarray(a, np.float64).ravel()
    assert a.size % 32 == 0
    q = np.empty(a.size, np.uint8)
    sf = np.empty(a.size // 32, np.uint8)
    deq = np.empty(a.size, np.float64)
    _load().oracle_mx_quantize(_ptr(a), a.size, _ptr(q), _ptr(sf), _ptr(deq))
    return q, sf, deq


def nv4_quantize(a: np.ndarray, gs: float):
    """Per-16 NVFP4 quantization of a 1-D array with global scale gs; returns
    (packed codes, e4m3 scale bytes, dequantized)."""
    a = np.ascontiguousarray(a, np.float64).ravel()
    assert a.size % 16 == 0
    q = np.zeros(a.size // 2, np.uint8)
    sf = np.empty(a.size // 16, np.uint8)
    deq = np.empty(a.size, np.float64)
    _load().oracle_nv4_quantize(_ptr(a), a.size, float(gs), _ptr(q), _ptr(sf), _ptr(deq))
    return q, sf, deq


# ---------------------------------------------------------------- routing
def route(topk_ids: np.ndarray, E: int, pad: int = 128):
    """Counting-sort routing.  Returns dict with counts, offsets (E+1),
    slot_of_pair, pad_offsets (E+1) and pad_slot_of_pair (all int64)."""
    ids = np.ascontiguousarray(topk_ids, np.int32)
    T, k = ids.shape
    P = T * k
    out = dict(counts=np.zeros(E, np.int64), offsets=np.zeros(E + 1, np.int64),
               slot_of_pair=np.zeros(P, np.int64), pad_offsets=np.zeros(E + 1, np.int64),
               pad_slot_of_pair=np.zeros(P, np.int64))
    rc = _load().oracle_route(T, E, k, _ptr(ids), pad, _ptr(out["counts"]), _ptr(out["offsets"]),
                              _ptr(out["slot_of_pair"]), _ptr(out["pad_offsets"]), _ptr(out["pad_slot_of_pair"]))
    if rc != 0:
        raise ValueError("expert id out of range")
    return out


# ---------------------------------------------------------------- router
def router_topk(logits: np.ndarray, k: int):
    """Top-k experts per token (decreasing logit, ties to the lower id) and the
    softmax of their logits in fp64.  ``logits`` is float32 [T, E].  Returns
    (ids int32 [T, k], weights float64 [T, k])."""
    lg = np.ascontiguousarray(logits, np.float32)
    T, E = lg.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    if _load().oracle_router_topk(T, E, int(k), _ptr(lg), _ptr(ids), _ptr(w)) != 0:
        raise ValueError("router_topk: k must lie in [1, E]")
    return ids, w


# ---------------------------------------------------------------- forward
def moe_ffn(x, w1, w2, topk_ids, topk_w, *, act=ACT_BF16, x_sf=None, w1_sf=None, w2_sf=None,
            tokens=None, threads: int = 0, swiglu_limit: float = 0.0, fp4_weights: bool = False) -> np.ndarray:
    """fp64 forward pass.

    bf16 inputs are uint16 bit patterns; MXFP8 inputs are uint8 e4m3 codes with
    uint8 e8m0 scale arrays (one per 32 along the last dimension).  Returns
    float64 out[n_tokens, D] for ``tokens`` (or all T tokens).  ``swiglu_limit``
    > 0 selects the clamped SwiGLU (gate <= limit, |up| <= limit).
    ``fp4_weights``: W1 [E, 2H, D/2] and W2 [E, D, H/2] hold MXFP4 weights
    (E2M1 codes packed two to a byte, low four bits first, one e8m0 scale per
    32 elements), x stays MXFP8.
    """
    mx = x_sf is not None
    x = np.ascontiguousarray(x)
    w1 = np.ascontiguousarray(w1)
    w2 = np.ascontiguousarray(w2)
    ids = np.ascontiguousarray(topk_ids, np.int32)
    tw = np.ascontiguousarray(topk_w, np.float32)
    T, D = x.shape
    E, H2, D1 = w1.shape
    H = H2 // 2
    k = ids.shape[1]
    if fp4_weights:
        assert mx and D1 * 2 == D and w2.shape == (E, D, H // 2) and tw.shape == ids.shape == (T, k)
    else:
        assert D1 == D and w2.shape == (E, D, H) and tw.shape == ids.shape == (T, k)
    if mx:
        x_sf, w1_sf, w2_sf = (np.ascontiguousarray(a, np.uint8) for a in (x_sf, w1_sf, w2_sf))
        assert x.dtype == np.uint8 and w1.dtype == np.uint8 and w2.dtype == np.uint8
    else:
        assert x.dtype == np.uint16 and w1.dtype == np.uint16 and w2.dtype == np.uint16
    tok = None if tokens is None else np.ascontiguousarray(tokens, np.int32)
    n = T if tok is None else tok.size
    out = np.zeros((n, D), np.float64)
    rc = _load().oracle_moe_ffn(T, E, D, H, k, IN_MXFP4W if fp4_weights else (IN_MXFP8 if mx else IN_BF16),
                                _ptr(x), _ptr(x_sf), _ptr(w1), _ptr(w1_sf), _ptr(w2), _ptr(w2_sf),
                                _ptr(ids), _ptr(tw), act, _ptr(tok), n, _ptr(out), int(threads),
                                float(swiglu_limit))
    if rc != 0:
        raise ValueError(f"oracle_moe_ffn failed ({rc})")
    return out


def moe_ffn_nvfp4(x, x_sf, x_gs, w1, w1_sf, w1_gs, w2, w2_sf, w2_gs, topk_ids, topk_w, *, act=ACT_EXACT,
                  act_gs: float = 0.0, tokens=None, threads: int = 0, swiglu_limit: float = 0.0) -> np.ndarray:
    """fp64 forward pass with NVFP4 operands: packed E2M1 codes (two per byte,
    low four bits first), e4m3 scale bytes per 16 along the last dimension, a
    global scale for x and one per expert for W1 and W2.  ``act`` is
    ACT_EXACT, ACT_BF16 or ACT_NVFP4 (requantized with global scale
    ``act_gs``)."""
    x, x_sf, w1, w1_sf, w2, w2_sf = (np.ascontiguousarray(a, np.uint8) for a in (x, x_sf, w1, w1_sf, w2, w2_sf))
    w1_gs = np.ascontiguousarray(w1_gs, np.float32)
    w2_gs = np.ascontiguousarray(w2_gs, np.float32)
    ids = np.ascontiguousarray(topk_ids, np.int32)
    tw = np.ascontiguousarray(topk_w, np.float32)
    T, D = x.shape[0], x.shape[1] * 2
    E, H2 = w1.shape[0], w1.shape[1]
    H = H2 // 2
    k = ids.shape[1]
    assert w1.shape == (E, 2 * H, D // 2) and w2.shape == (E, D, H // 2)
    assert x_sf.shape == (T, D // 16) and w1_sf.shape == (E, 2 * H, D // 16) and w2_sf.shape == (E, D, H // 16)
    assert w1_gs.shape == (E,) and w2_gs.shape == (E,) and tw.shape == ids.shape == (T, k)
    tok = None if tokens is None else np.ascontiguousarray(tokens, np.int32)
    n = T if tok is None else tok.size
    out = np.zeros((n, D), np.float64)
    rc = _load().oracle_moe_ffn_nvfp4(T, E, D, H, k, _ptr(x), _ptr(x_sf), float(x_gs), _ptr(w1), _ptr(w1_sf),
                                      _ptr(w1_gs), _ptr(w2), _ptr(w2_sf), _ptr(w2_gs), _ptr(ids), _ptr(tw), act,
                                      float(act_gs), _ptr(tok), n, _ptr(out), int(threads), float(swiglu_limit))
    if rc != 0:
        raise ValueError(f"oracle_moe_ffn_nvfp4 failed ({rc})")
    return out


def max_threads() -> int:
    return _load().oracle_max_threads()
