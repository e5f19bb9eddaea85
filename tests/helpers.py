"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
run the library through its C ABI, compare against the CPU oracle."""
import numpy as np
import torch

import grouped_gemm_gb300 as moe

# parity tolerances of the path: max|gpu - ref| <= TOL_MAX * max|ref| and
# sum|gpu - ref| / sum|ref| <= TOL_MEAN (ratio of L1 norms)
TOL = {"bf16": (2e-2, 5e-3), "mxfp8": (4e-2, 1e-2)}


def to_dev(inp, device="cuda"):
    d = {}
    for key in ("x", "w1", "w2"):
        a = inp[key]
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        d[key] = t.to(device)
    for key in ("x_sf", "w1_sf", "w2_sf"):
        if key in inp:
            d[key] = torch.from_numpy(inp[key]).to(device)
    d["topk_ids"] = torch.from_numpy(np.ascontiguousarray(inp["topk_ids"], np.int32)).to(device)
    d["topk_w"] = torch.from_numpy(np.ascontiguousarray(inp["topk_w"], np.float32)).to(device)
    return d


def run_forward(inp, dev, pipeline=moe.MOE_SPLIT, dtype=moe.MOE_BF16, workspace=None, out=None, check_status=True):
    w = inp["workload"]
    T, D, H, E, k = w.T, w.D, w.H, w.E, w.k
    if out is None:
        out = torch.full((T, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    if workspace is None:
        workspace = moe.alloc_workspace(T, E, D, H, k, dtype, pipeline)
    moe.moe_ffn_forward(dev["x"], dev["w1"], dev["w2"], dev["topk_ids"], dev["topk_w"], out, E=E, D=D, H=H, k=k,
                        workspace=workspace, dtype=dtype, pipeline=pipeline, x_sf=dev.get("x_sf"),
                        w1_sf=dev.get("w1_sf"), w2_sf=dev.get("w2_sf"), T=T)
    if check_status:
        st = moe.moe_ffn_sync_status(workspace)
        assert st == 0, moe.moe_ffn_status_string(st)
    return out, workspace


def compare(gpu, ref, dtype="bf16"):
    """Return (max_rel, mean_rel, cosine) of gpu vs the fp64 reference."""
    g = gpu.float().cpu().double().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape
    assert np.isfinite(g).all(), "non-finite output"
    diff = np.abs(g - r)
    max_rel = diff.max() / max(np.abs(r).max(), 1e-30)
    mean_rel = diff.sum() / max(np.abs(r).sum(), 1e-30)
    cos = float((g * r).sum() / max(np.sqrt((g * g).sum() * (r * r).sum()), 1e-30))
    return max_rel, mean_rel, cos


def assert_close(gpu, ref, dtype="bf16", label="", tol=None):
    max_rel, mean_rel, cos = compare(gpu, ref, dtype)
    tmax, tmean = TOL[dtype] if tol is None else tol
    msg = f"{label}: max_rel={max_rel:.3e} (<= {tmax}) mean_rel={mean_rel:.3e} (<= {tmean}) cos={cos:.6f}"
    assert max_rel <= tmax and mean_rel <= tmean, msg
    return max_rel, mean_rel, cos


def coverage_tokens(topk_ids, n_random=1000, seed=1, pad=128):
    """A deterministic sample of tokens for checking a full-size output on the
    oracle: for every expert with routed pairs, the tokens of its first and
    last routed row and of the first row of its last 128-row block (the tail
    block, which in the CTA-pair kernels may be the odd half pair), plus
    n_random tokens drawn with a seeded generator.  Sorted, distinct, int32.
    Row order within an expert follows the flat pair index t*k + j."""
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    flat = ids.ravel()
    order = np.argsort(flat, kind="stable")          # pairs grouped by expert, flat order within
    experts, starts, counts = np.unique(flat[order], return_index=True, return_counts=True)
    picks = []
    for s, n in zip(starts, counts):
        ranks = {0, n - 1, (n - 1) // pad * pad}
        picks.extend(order[s + r] // k for r in ranks)
    rnd = np.random.default_rng(seed).choice(T, min(T, n_random), replace=False)
    return np.unique(np.concatenate([np.asarray(picks, np.int64), rnd])).astype(np.int32)


_INPUT_CACHE = {}


def cached_inputs(name, seed=0):
    """wl.make_inputs(name, seed), kept for the next test that asks (the large
    workloads take seconds to draw).  Callers must not modify the arrays."""
    from grouped_gemm_gb300 import workloads as wl
    key = (name, seed)
    if key not in _INPUT_CACHE:
        if len(_INPUT_CACHE) >= 2:
            _INPUT_CACHE.pop(next(iter(_INPUT_CACHE)))
        _INPUT_CACHE[key] = wl.make_inputs(name, seed=seed)
    return _INPUT_CACHE[key]
