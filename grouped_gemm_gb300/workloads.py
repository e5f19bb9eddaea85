"""Seeded synthetic inputs for the routed MoE SwiGLU FFN forward pass.

This module only draws inputs; it holds none of the forward pass's arithmetic,
so both the CUDA path and the CPU oracle can consume the same bytes.

Five named workloads, with the shapes and distributions of the problem the
"Prime Flash MoE" and Pearl "Optimizing Grouped GEMM for MoE on Blackwell"
pages discuss (x ~ N(0,1), weights ~ N(0, 0.02^2), top-k routing with
softmax-normalized weights over the selected experts):

  tiny          T=64     D=256  H=128  E=8   k=2  top-2 of N(0,1) router logits
  decode        T=64     D=6144 H=2048 E=32  k=8  uniform distinct experts
  prefill       T=4096   D=2048 H=768  E=128 k=8  top-8 of N(0,1) router logits
  large_skewed  T=131072 D=2048 H=768  E=128 k=8  Zipf(1.1) expert popularity
  mxfp8         T=16384  D=4096 H=1536 E=64  k=8  uniform distinct, MXFP8 inputs

Arrays are numpy: bf16 as uint16 bit patterns, MXFP8 as uint8 e4m3 codes with
uint8 e8m0 scale bytes (one per 32 elements along the contiguous dimension).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    H: int
    E: int
    k: int
    routing: str          # "topk_logits" | "uniform" | "zipf"
    dtype: str = "bf16"   # "bf16" | "mxfp8" | "mxfp4w" (MXFP8 activations, MXFP4 weights) | "nvfp4"

    @property
    def pairs(self) -> int:
        return self.T * self.k

    @property
    def flops(self) -> int:
        """Multiply-adds x 2 of the three projections per routed pair."""
        return 6 * self.T * self.k * self.D * self.H


WORKLOADS = {
    "tiny": Workload("tiny", 64, 256, 128, 8, 2, "topk_logits"),
    "decode": Workload("decode", 64, 6144, 2048, 32, 8, "uniform"),
    "prefill": Workload("prefill", 4096, 2048, 768, 128, 8, "topk_logits"),
    "large_skewed": Workload("large_skewed", 131072, 2048, 768, 128, 8, "zipf"),
    "mxfp8": Workload("mxfp8", 16384, 4096, 1536, 64, 8, "uniform", "mxfp8"),
    # the decode shape with MXFP4 expert weights (MXFP8 activations)
    "decode_mxfp4w": Workload("decode_mxfp4w", 64, 6144, 2048, 32, 8, "uniform", "mxfp4w"),
    # the decode shape with NVFP4 activations and weights
    "decode_nvfp4": Workload("decode_nvfp4", 64, 6144, 2048, 32, 8, "uniform", "nvfp4"),
}

ZIPF_S = 1.1
ZIPF_ZERO_EXPERTS = 8   # least popular ranks held at popularity 0


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (torch's round-to-nearest-even cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def _softmax_rows(logits: np.ndarray) -> np.ndarray:
    z = logits.astype(np.float64)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    return (p / p.sum(axis=1, keepdims=True)).astype(np.float32)


def draw_routing(rng: np.random.Generator, T: int, E: int, k: int, kind: str):
    """Return (topk_ids int32 [T,k], topk_w float32 [T,k])."""
    if kind == "topk_logits":
        logits = rng.standard_normal(size=(T, E))
        # descending by logit, ties to the lower expert id (stable sort)
        order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
        sel = np.take_along_axis(logits, order, axis=1)
        return order.astype(np.int32), _softmax_rows(sel)
    if kind == "uniform":
        keys = rng.random(size=(T, E))
        ids = np.argsort(keys, axis=1, kind="stable")[:, :k]
        return ids.astype(np.int32), _softmax_rows(rng.standard_normal(size=(T, k)))
    if kind == "zipf":
        # Zipf(s) popularity over the E - ZIPF_ZERO_EXPERTS most popular ranks,
        # ranks assigned to experts by a seeded permutation; distinct experts per
        # token drawn without replacement via Gumbel-top-k on log popularity.
        nz = E - ZIPF_ZERO_EXPERTS
        pop = np.zeros(E)
        pop[:nz] = np.arange(1, nz + 1, dtype=np.float64) ** (-ZIPF_S)
        perm = rng.permutation(E)
        p_expert = np.empty(E)
        p_expert[perm] = pop
        logp = np.full(E, -np.inf)
        logp[p_expert > 0] = np.log(p_expert[p_expert > 0])
        ids = np.empty((T, k), np.int32)
        chunk = 16384
        for t0 in range(0, T, chunk):
            n = min(chunk, T - t0)
            g = -np.log(-np.log(rng.random(size=(n, E)) + 1e-300) + 1e-300)
            keys = logp[None, :] + g
            ids[t0:t0 + n] = np.argsort(-keys, axis=1, kind="stable")[:, :k]
        return ids, _softmax_rows(rng.standard_normal(size=(T, k)))
    raise ValueError(kind)


def router_logits(T: int, E: int, seed: int = 0) -> np.ndarray:
    """float32 router logits [T, E] ~ N(0, 1), one per (token, expert)."""
    return np.random.default_rng(seed).standard_normal(size=(T, E), dtype=np.float32)


def mx_encode_rows(a: np.ndarray):
    """Encode float32 rows (last dim a multiple of 32) as e4m3 codes + e8m0 scales.

    Input preparation only: each block's scale 2^e is the smallest power of two
    with max|a|/2^e <= 448, and the codes come from torch's float8_e4m3fn cast.
    """
    a = np.ascontiguousarray(a, np.float32)
    shp = a.shape
    blk = a.reshape(-1, 32)
    amax = np.abs(blk).max(axis=1).astype(np.float64)
    f, ex = np.frexp(amax)                       # amax = f 2^ex, f in [0.5, 1)
    e = (ex - 1) - 8 + ((2.0 * f) > 1.75)
    e = np.where(amax == 0, 0, e).astype(np.int64)
    scaled = (blk.astype(np.float64) * np.ldexp(1.0, -e)[:, None]).astype(np.float32)
    q = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    sf = (e + 127).astype(np.uint8)
    return q.reshape(shp), sf.reshape(shp[:-1] + (shp[-1] // 32,))


_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def mx4_encode_rows(a: np.ndarray):
    """Encode float32 rows (last dim a multiple of 32) as MXFP4: E2M1 codes
    packed two to a byte (element 2j in the low four bits of byte j) + e8m0
    scales, one per 32 elements.

    Input preparation only: each block's scale 2^e is the smallest power of two
    with max|a|/2^e <= 6; each scaled value goes to the nearest grid point of
    |E2M1| (ties to the even code), with its sign.
    """
    a = np.ascontiguousarray(a, np.float32)
    shp = a.shape
    blk = a.reshape(-1, 32).astype(np.float64)
    amax = np.abs(blk).max(axis=1)
    f, ex = np.frexp(amax)
    e = (ex - 1) - 2 + ((2.0 * f) > 1.5)
    e = np.where(amax == 0, 0, e).astype(np.int64)
    scaled = blk * np.ldexp(1.0, -e)[:, None]
    mag = np.minimum(np.abs(scaled), 6.0)
    dist = np.abs(mag[..., None] - _E2M1_GRID)                   # distance to each grid point
    best = dist.min(axis=-1, keepdims=True)
    tied = np.isclose(dist, best, rtol=0, atol=0)
    # among the nearest points prefer the even code (codes 0, 2, 4, 6 = grid points 0, 1, 2, 4)
    even = (np.arange(8) % 2 == 0)
    code = np.where((tied & even).any(axis=-1), np.argmax(tied & even, axis=-1), np.argmax(tied, axis=-1))
    code = code.astype(np.uint8) | np.where(scaled < 0, 8, 0).astype(np.uint8)
    code = code.reshape(shp)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    sf = (e + 127).astype(np.uint8).reshape(shp[:-1] + (shp[-1] // 32,))
    return packed, sf


E4M3_MAX = 448.0
E2M1_MAX = 6.0


def nv4_global_scale(a: np.ndarray) -> np.float32:
    """Global scale of an NVFP4 tensor: amax / (448 * 6), so that the largest
    block scale is the largest e4m3 value (1.0 for an all-zero tensor)."""
    amax = float(np.abs(a).max()) if a.size else 0.0
    return np.float32(amax / (E4M3_MAX * E2M1_MAX) if amax > 0 else 1.0)


def nv4_encode_rows(a: np.ndarray, gs: float):
    """Encode float32 rows (last dim a multiple of 16) as NVFP4 with global
    scale gs: E2M1 codes packed two to a byte (element 2j in the low four
    bits) + e4m3 scale bytes, one per 16 elements.

    Input preparation only: each block's scale is torch's float8_e4m3fn cast
    of amax / (6 gs), clamped to 448 first; each element goes to the nearest E2M1 value of
    a / (scale gs) (ties to the even code, saturating at 6).
    """
    a = np.ascontiguousarray(a, np.float32)
    shp = a.shape
    blk = a.reshape(-1, 16).astype(np.float64)
    amax = np.abs(blk).max(axis=1)
    # torch's cast does not saturate (above 464 it gives NaN): clamp to 448 first
    ratio = np.minimum(amax / (E2M1_MAX * float(gs)), E4M3_MAX)
    sfc = torch.from_numpy(ratio.astype(np.float32)).to(torch.float8_e4m3fn)
    sval = sfc.double().numpy()
    sf = sfc.view(torch.uint8).numpy()
    denom = sval * float(gs)
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = np.where(denom[:, None] > 0, blk / denom[:, None], 0.0)
    mag = np.minimum(np.abs(scaled), E2M1_MAX)
    dist = np.abs(mag[..., None] - _E2M1_GRID)
    best = dist.min(axis=-1, keepdims=True)
    tied = dist == best
    even = (np.arange(8) % 2 == 0)
    code = np.where((tied & even).any(axis=-1), np.argmax(tied & even, axis=-1), np.argmax(tied, axis=-1))
    code = code.astype(np.uint8) | np.where(scaled < 0, 8, 0).astype(np.uint8)
    code = code.reshape(shp)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    return packed, sf.reshape(shp[:-1] + (shp[-1] // 16,))


def make_inputs(w: Workload | str, seed: int = 0, T: int | None = None):
    """Draw one workload's inputs.  Order of draws: x, W1, W2, routing.

    ``T`` overrides the token count (routing draws for the smaller T), used for
    sampled checks.  Returns a dict of numpy arrays plus the Workload.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    if T is not None:
        w = dataclasses.replace(w, T=T)
    rng = np.random.default_rng(seed)
    out = {"workload": w}
    if w.dtype == "bf16":
        out["x"] = _bf16_bits(_normal(rng, (w.T, w.D), 1.0))
        w1 = np.empty((w.E, 2 * w.H, w.D), np.uint16)
        for e in range(w.E):
            w1[e] = _bf16_bits(_normal(rng, (2 * w.H, w.D), 0.02))
        w2 = np.empty((w.E, w.D, w.H), np.uint16)
        for e in range(w.E):
            w2[e] = _bf16_bits(_normal(rng, (w.D, w.H), 0.02))
        out["w1"], out["w2"] = w1, w2
    elif w.dtype == "nvfp4":  # NVFP4 activations and weights, global scales per tensor / per expert
        xa = _normal(rng, (w.T, w.D), 1.0)
        out["x_gs"] = nv4_global_scale(xa)
        out["x"], out["x_sf"] = nv4_encode_rows(xa, out["x_gs"])
        for name, rows, cols in (("w1", 2 * w.H, w.D), ("w2", w.D, w.H)):
            q = np.empty((w.E, rows, cols // 2), np.uint8)
            sf = np.empty((w.E, rows, cols // 16), np.uint8)
            gs = np.empty(w.E, np.float32)
            for e in range(w.E):
                a = _normal(rng, (rows, cols), 0.02)
                gs[e] = nv4_global_scale(a)
                q[e], sf[e] = nv4_encode_rows(a, gs[e])
            out[name], out[name + "_sf"], out[name + "_gs"] = q, sf, gs
        # global scale of act (a calibrated constant of the model, not drawn):
        # gate and up have standard deviation 0.02 sqrt(D) for these draws, so
        # act blocks up to 25 (0.02^2 D) keep their e4m3 scale below 448
        out["act_gs"] = np.float32(25.0 * 0.02 ** 2 * w.D / (6.0 * 448.0))
    elif w.dtype == "mxfp4w":  # MXFP8 activations, MXFP4 weights
        out["x"], out["x_sf"] = mx_encode_rows(_normal(rng, (w.T, w.D), 1.0))
        w1 = np.empty((w.E, 2 * w.H, w.D // 2), np.uint8)
        w1_sf = np.empty((w.E, 2 * w.H, w.D // 32), np.uint8)
        for e in range(w.E):
            w1[e], w1_sf[e] = mx4_encode_rows(_normal(rng, (2 * w.H, w.D), 0.02))
        w2 = np.empty((w.E, w.D, w.H // 2), np.uint8)
        w2_sf = np.empty((w.E, w.D, w.H // 32), np.uint8)
        for e in range(w.E):
            w2[e], w2_sf[e] = mx4_encode_rows(_normal(rng, (w.D, w.H), 0.02))
        out.update(w1=w1, w1_sf=w1_sf, w2=w2, w2_sf=w2_sf)
    else:
        out["x"], out["x_sf"] = mx_encode_rows(_normal(rng, (w.T, w.D), 1.0))
        w1 = np.empty((w.E, 2 * w.H, w.D), np.uint8)
        w1_sf = np.empty((w.E, 2 * w.H, w.D // 32), np.uint8)
        for e in range(w.E):
            w1[e], w1_sf[e] = mx_encode_rows(_normal(rng, (2 * w.H, w.D), 0.02))
        w2 = np.empty((w.E, w.D, w.H), np.uint8)
        w2_sf = np.empty((w.E, w.D, w.H // 32), np.uint8)
        for e in range(w.E):
            w2[e], w2_sf[e] = mx_encode_rows(_normal(rng, (w.D, w.H), 0.02))
        out.update(w1=w1, w1_sf=w1_sf, w2=w2, w2_sf=w2_sf)
    out["topk_ids"], out["topk_w"] = draw_routing(rng, w.T, w.E, w.k, w.routing)
    return out


def make_custom(T: int, D: int, H: int, E: int, k: int, seed: int = 0, routing: str = "topk_logits",
                dtype: str = "bf16"):
    """Inputs for an arbitrary shape with the same distributions (test cases)."""
    return make_inputs(Workload("custom", T, D, H, E, k, routing, dtype), seed=seed)
