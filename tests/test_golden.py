"""The oracle's codecs against format facts the pages state
(tests/golden/format_facts.txt, each fact with its page and section).  CPU only."""
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def facts():
    out = {}
    with open(os.path.join(HERE, "golden", "format_facts.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *vals = line.split()
                out[key] = [float(v) for v in vals]
    return out


F = facts()


def test_e4m3_largest_value():
    assert oracle.e4m3_to_f64(oracle.f64_to_e4m3(1e9))[()] == F["e4m3_max"][0]
    finite = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))   # 0x7F is NaN
    assert finite.max() == F["e4m3_max"][0]


def test_mx_blocks():
    n = 4 * int(F["mx_block"][0])
    q, sf, _ = oracle.mx_quantize(np.linspace(-1, 1, n))
    assert sf.size == n // F["mx_block"][0]
    # MXFP4 shares the MX block length
    assert F["mxfp4_block"][0] == F["mx_block"][0]


def test_e2m1_is_four_bits_with_max_six():
    codes = np.arange(2 ** int(F["e2m1_bits"][0]), dtype=np.uint8)
    vals = oracle.e2m1_to_f64(codes)
    assert np.abs(vals).max() == F["nvfp4_scale_divisor"][0]
    # the encoder never emits a code outside four bits
    assert oracle.f64_to_e2m1(np.linspace(-100, 100, 1001)).max() < 2 ** int(F["e2m1_bits"][0])


def test_nvfp4_block_and_scale_rule():
    block = 256 // int(F["nvfp4_scales_per_256"][0])
    n = 4 * block
    q, sf, _ = oracle.nv4_quantize(np.linspace(-3, 3, n), 1.0)
    assert sf.size == n // block and q.size == n // 2
    # a block whose amax is divisor * s (s an e4m3 value) gets the scale s
    for s in (0.25, 1.0, 1.125, 40.0):
        v = np.zeros(block)
        v[3] = -F["nvfp4_scale_divisor"][0] * s
        _, sfb, deq = oracle.nv4_quantize(v, 1.0)
        assert oracle.e4m3_to_f64(sfb)[0] == s and deq[3] == v[3]
