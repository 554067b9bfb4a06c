"""The FMA-pipe exp2 used for part of the forward's probabilities
(exp2_poly2 in csrc/sm100_ptx.cuh): its constants are the ones the Remez fit
in csrc/gen_exp2_poly.py produces, and the method (round-to-nearest split,
cubic for 2^f, exponent add) stays within its stated relative error bound
over the clamped range [-125, 8], emulated step by step in fp32."""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "softmax_attention_numerics_gb300", "csrc")


def kernel_coeffs():
    text = open(os.path.join(CSRC, "sm100_ptx.cuh")).read()
    body = text[text.index("float2 exp2_poly2"):]
    body = body[:body.index("return make_float2")]
    vals = []
    for v in re.findall(r"([0-9]\.[0-9]+e[-+][0-9]+)f", body):
        if float(v) not in vals:
            vals.append(float(v))
    # order of first appearance: c3, c2, c1, c0
    return vals[0], vals[1], vals[2], vals[3]


def test_constants_match_the_fit():
    import importlib.util
    spec = importlib.util.spec_from_file_location("gen", os.path.join(CSRC, "gen_exp2_poly.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    c, err = gen.remez_exp2()
    assert err < 1e-4
    c3, c2, c1, c0 = kernel_coeffs()
    assert np.allclose([c0, c1, c2, c3], np.float32(c), rtol=1e-6, atol=0)


def emulate(x):
    f32 = np.float32
    c3, c2, c1, c0 = (f32(v) for v in kernel_coeffs())
    x = np.minimum(np.maximum(x.astype(f32), f32(-125.0)), f32(8.0))
    t = (x + f32(12582912.0)).astype(f32)
    nr = (t - f32(12582912.0)).astype(f32)
    f = (x - nr).astype(f32)
    q = (c3 * f + c2).astype(f32)
    q = (q * f + c1).astype(f32)
    q = (q * f + c0).astype(f32)
    bits = q.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_relative_error_over_clamped_range():
    x = np.concatenate([np.linspace(-125, 8, 2_000_001), np.arange(-125, 9) + 0.5,
                        np.arange(-125, 9).astype(np.float64)])
    got = emulate(x).astype(np.float64)
    ref = np.exp2(np.clip(x.astype(np.float32).astype(np.float64), -125, 8))
    rel = np.abs(got - ref) / ref
    assert rel.max() < 1.2e-4          # fit bound 7.5e-5 plus fp32 rounding of the steps


def test_below_range_is_tiny_and_positive():
    got = emulate(np.array([-126.0, -200.0, -1e30, -np.inf]))
    assert np.all(got > 0) and np.all(got <= 2.0 ** -124)
