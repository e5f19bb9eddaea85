"""The forward pass with its extras (moe_ffn_forward_ex) against the oracle:
the clamped SwiGLU ("Porting Block-Scaled GEMM Kernels from Blackwell to
Rubin" sec. 5.3: gate clamped from above, up on both sides), shared experts
run on every token ("GC-MoE on SM120" sec. 4.7), and both together with the
router.  Every kernel family's SwiGLU epilogue is covered: single-CTA and
CTA-pair split GEMMs, the fused pipeline on clusters and with split-K, and
both MXFP8 pipelines.  Parity tolerances (bf16 2e-2 / 5e-3, MXFP8 4e-2 /
1e-2); the oracle gets the same extended ids and weights, built here with
numpy (routed ids, then E .. E + n_shared - 1 at weight 1)."""
import numpy as np
import pytest
import torch

import grouped_gemm_gb300 as moe
import oracle
from grouped_gemm_gb300 import workloads as wl

from helpers import assert_close, to_dev

pytestmark = pytest.mark.gpu

MODES = {  # name: (pipeline, options)
    "split": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 0, moe.MOE_OPT_TILE_M: 128}),
    "split_pair2": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 1}),
    "split_wide": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 1, moe.MOE_OPT_WIDE_UP: 1}),
    "split_m64": (moe.MOE_SPLIT, {moe.MOE_OPT_PAIR_MMA: 0, moe.MOE_OPT_TILE_M: 64}),
    "fused": (moe.MOE_FUSED, {}),
    "fused_dsmem": (moe.MOE_FUSED, {moe.MOE_OPT_FUSED_DSMEM: 1}),
    "fused_splitk": (moe.MOE_FUSED, {moe.MOE_OPT_FUSED_CLUSTER: 0}),
}
DEFAULTS = {moe.MOE_OPT_PAIR_MMA: 2, moe.MOE_OPT_FUSED_CLUSTER: 1, moe.MOE_OPT_WIDE_UP: 0, moe.MOE_OPT_TILE_M: 0, moe.MOE_OPT_FUSED_DSMEM: 0}


def extended(ids, tw, E, ns):
    T = ids.shape[0]
    if ns == 0:
        return ids, tw
    return (np.concatenate([ids, np.tile(np.arange(E, E + ns, dtype=np.int32), (T, 1))], axis=1),
            np.concatenate([tw, np.ones((T, ns), np.float32)], axis=1))


def run_ex(inp, E, k, ns, limit, pipeline, dtype=moe.MOE_BF16, logits=None, dev=None, w1p=None, w2p=None):
    w = inp["workload"]
    dev = dev or to_dev(inp)
    T, D, H = w.T, w.D, w.H
    ids = dev["topk_ids"][:, :k].contiguous() if logits is None else torch.empty(T, k, dtype=torch.int32, device="cuda")
    tw = dev["topk_w"][:, :k].contiguous() if logits is None else torch.empty(T, k, device="cuda")
    out = torch.full((T, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(T, E, D, H, k, dtype, pipeline, n_shared=ns)
    moe.moe_ffn_forward_ex(dev["x"], dev["w1"], dev["w2"], ids, tw, out, E=E, D=D, H=H, k=k, workspace=ws,
                           dtype=dtype, pipeline=pipeline, x_sf=dev.get("x_sf"), w1_sf=w1p, w2_sf=w2p,
                           swiglu_limit=limit, n_shared=ns,
                           router_logits=None if logits is None else torch.from_numpy(logits).cuda())
    assert moe.moe_ffn_sync_status(ws) == 0
    return out, ids.cpu().numpy(), tw.cpu().numpy()


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("T,D,H,E,k,ns,limit", [
    (200, 512, 256, 8, 2, 0, 0.25),     # clamp only
    (300, 512, 256, 16, 4, 1, 0.0),     # one shared expert
    (700, 512, 256, 8, 2, 2, 0.3),      # two shared experts and the clamp; shared experts of 700 rows
    (1000, 2048, 768, 16, 4, 1, 0.5),   # prefill dims
])
def test_forward_ex(mode, T, D, H, E, k, ns, limit):
    inp = wl.make_custom(T, D, H, E + ns, k, seed=T + ns, routing="uniform")
    ids = inp["topk_ids"] % E                      # routed experts only
    inp["topk_ids"] = ids
    pipeline, opts = MODES[mode]
    for o, v in opts.items():
        moe.moe_ffn_set_option(o, v)
    try:
        out, _, _ = run_ex(inp, E, k, ns, limit, pipeline)
    finally:
        for o in opts:
            moe.moe_ffn_set_option(o, DEFAULTS[o])
    ide, twe = extended(ids, inp["topk_w"], E, ns)
    ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], ide, twe, act=oracle.ACT_BF16, swiglu_limit=limit)
    if limit > 0:  # the clamp must be active for a real share of the gates
        plain = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], ide, twe, act=oracle.ACT_BF16)
        assert np.abs(plain - ref).sum() > 0.02 * np.abs(ref).sum()
    assert_close(out, ref, label=f"{mode} T={T} E={E} ns={ns} limit={limit}")


@pytest.mark.parametrize("pipeline", [moe.MOE_SPLIT, moe.MOE_FUSED])
def test_forward_ex_router_shared_and_clamp(pipeline):
    T, D, H, E, k, ns, limit = 400, 512, 256, 12, 3, 1, 0.3
    inp = wl.make_custom(T, D, H, E + ns, k, seed=31, routing="uniform")
    lg = wl.router_logits(T, E, seed=32)
    out, gids, gw = run_ex(inp, E, k, ns, limit, pipeline, logits=lg)
    rids, rw = oracle.router_topk(lg, k)
    assert np.array_equal(gids, rids)
    ide, twe = extended(rids, rw.astype(np.float32), E, ns)
    ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], ide, twe, act=oracle.ACT_BF16, swiglu_limit=limit)
    assert_close(out, ref, label="router + shared + clamp")


@pytest.mark.parametrize("pipeline", [moe.MOE_SPLIT, moe.MOE_FUSED])
def test_forward_ex_mxfp8(pipeline):
    T, D, H, E, k, ns, limit = 300, 512, 256, 8, 2, 1, 0.25
    inp = wl.make_custom(T, D, H, E + ns, k, seed=41, routing="uniform", dtype="mxfp8")
    inp["topk_ids"] = inp["topk_ids"] % E
    dev = to_dev(inp)
    w1p = torch.empty(inp["w1_sf"].size, dtype=torch.uint8, device="cuda")
    w2p = torch.empty(inp["w2_sf"].size, dtype=torch.uint8, device="cuda")
    moe.moe_ffn_prepare_mxfp8_weights(dev["w1_sf"], dev["w2_sf"], w1p, w2p, E + ns, D, H)
    out, _, _ = run_ex(inp, E, k, ns, limit, pipeline, dtype=moe.MOE_MXFP8, dev=dev, w1p=w1p, w2p=w2p)
    ide, twe = extended(inp["topk_ids"], inp["topk_w"], E, ns)
    ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], ide, twe, act=oracle.ACT_MXFP8, x_sf=inp["x_sf"],
                         w1_sf=inp["w1_sf"], w2_sf=inp["w2_sf"], swiglu_limit=limit)
    assert_close(out, ref, dtype="mxfp8", label=f"mxfp8 pipeline={pipeline} shared + clamp")


def test_forward_ex_rejects_bad_extras():
    inp = wl.make_custom(8, 256, 128, 4, 2, seed=1)
    dev = to_dev(inp)
    out = torch.empty(8, 256, dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(8, 4, 256, 128, 2)
    for kw in ({"swiglu_limit": -1.0}, {"n_shared": -1}, {"n_shared": 1021}):
        assert moe.moe_ffn_forward_ex(dev["x"], dev["w1"], dev["w2"], dev["topk_ids"], dev["topk_w"], out, E=4, D=256,
                                      H=128, k=2, workspace=ws, check=False, **kw) == 1
    # a workspace sized without the shared expert is too small for one
    assert moe.moe_ffn_forward_ex(dev["x"], dev["w1"], dev["w2"], dev["topk_ids"], dev["topk_w"], out, E=3, D=256,
                                  H=128, k=2, workspace=ws, n_shared=1, check=False) == 5


@pytest.mark.parametrize("pipeline", [moe.MOE_SPLIT, moe.MOE_FUSED])
def test_forward_ex_routed_id_of_a_shared_expert_is_bad_routing(pipeline):
    # With one shared expert the extended problem has E + 1 experts, but a
    # routed id must still lie in [0, E): id E names the shared expert and is
    # reported as a bad id (the pair dropped), not run as that expert.
    T, D, H, E, k, ns = 64, 256, 128, 4, 2, 1
    inp = wl.make_custom(T, D, H, E + ns, k, seed=17, routing="uniform")
    ids = inp["topk_ids"] % E
    ids[9, 1] = E
    inp["topk_ids"] = ids
    dev = to_dev(inp)
    out = torch.full((T, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(T, E, D, H, k, moe.MOE_BF16, pipeline, n_shared=ns)
    moe.moe_ffn_forward_ex(dev["x"], dev["w1"], dev["w2"], dev["topk_ids"], dev["topk_w"], out, E=E, D=D, H=H, k=k,
                           workspace=ws, pipeline=pipeline, n_shared=ns)
    assert moe.moe_ffn_sync_status(ws) == 4          # MOE_ERR_BAD_ROUTING
    kept = ids.copy()
    tw = inp["topk_w"].copy()
    kept[9, 1] = 0
    tw[9, 1] = 0.0
    ide, twe = extended(kept, tw, E, ns)
    ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], ide, twe, act=oracle.ACT_BF16)
    assert_close(out, ref, label="routed id E dropped")
