"""The seeded input recipe: routing structure and value distributions of the
workloads (CPU only; the draws, not the method)."""
import numpy as np
import torch

from grouped_gemm_gb300 import workloads as wl


def test_zipf_routing_has_empty_and_skewed_experts():
    w = wl.WORKLOADS["large_skewed"]
    ids, tw = wl.draw_routing(np.random.default_rng(0), 16384, w.E, w.k, "zipf")
    counts = np.bincount(ids.ravel(), minlength=w.E)
    assert (counts == 0).sum() == wl.ZIPF_ZERO_EXPERTS          # the least popular ranks never drawn
    live = counts[counts > 0]
    assert live.max() > 20 * live.min()                          # Zipf(1.1) skew
    assert all(len(set(r)) == w.k for r in ids)                  # k distinct experts per token
    np.testing.assert_allclose(tw.sum(axis=1), 1.0, rtol=1e-6)


def test_uniform_and_logit_routing():
    for kind in ("uniform", "topk_logits"):
        ids, tw = wl.draw_routing(np.random.default_rng(1), 4096, 32, 8, kind)
        assert ids.dtype == np.int32 and tw.dtype == np.float32
        assert all(len(set(r)) == 8 for r in ids)
        counts = np.bincount(ids.ravel(), minlength=32)
        assert counts.min() > 0.7 * counts.mean() and counts.max() < 1.3 * counts.mean()
        np.testing.assert_allclose(tw.sum(axis=1), 1.0, rtol=1e-6)
        assert (tw > 0).all()


def test_topk_logits_weights_follow_the_order():
    ids, tw = wl.draw_routing(np.random.default_rng(2), 256, 16, 4, "topk_logits")
    assert (np.diff(tw.astype(np.float64), axis=1) <= 1e-7).all()   # selected by decreasing logit


def test_value_distributions():
    inp = wl.make_custom(T=512, D=256, H=128, E=4, k=2, seed=3)
    f = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    x, w1 = f(inp["x"]), f(inp["w1"])
    assert abs(x.std() - 1.0) < 0.02 and abs(x.mean()) < 0.02
    assert abs(w1.std() - 0.02) < 0.001
    # same seed, same bytes
    again = wl.make_custom(T=512, D=256, H=128, E=4, k=2, seed=3)
    assert all(np.array_equal(inp[k], again[k]) for k in ("x", "w1", "w2", "topk_ids", "topk_w"))
