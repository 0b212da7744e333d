"""The FMA-pipe exp2 used for part of the softmax: its constants come from the
in-repo Remez fit, and its float32 evaluation (emulated bit for bit here)
stays within the stated error bound of the true 2^x."""
import os
import re

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "joint_attention_gb300", "csrc")


def header_coefficients():
    text = open(os.path.join(CSRC, "exp2_poly.h")).read()
    return [np.float32(float(v)) for v in re.findall(r"kExp2C\d = ([0-9.eE+-]+)f;", text)]


def emulate(x):
    """The kernel's exp2_poly in float32 numpy, operation for operation."""
    x = np.maximum(np.asarray(x, np.float32), np.float32(-125.0))
    c0, c1, c2, c3 = header_coefficients()
    t = (x + np.float32(12582912.0)).astype(np.float32)
    n = (t - np.float32(12582912.0)).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = (c3 * f + c2).astype(np.float32)
    p = (p * f + c1).astype(np.float32)
    p = (p * f + c0).astype(np.float32)
    bits = (p.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def test_header_matches_the_remez_fit():
    import importlib.util

    spec = importlib.util.spec_from_file_location("gen", os.path.join(CSRC, "gen_exp2_poly.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    coef, err = gen.remez(3)
    np.testing.assert_array_equal(np.asarray(header_coefficients()), coef.astype(np.float32))
    assert err < 8e-5


def test_relative_error_bound_over_the_softmax_range():
    # fused argument range of the softmax: (s - m) * scale * log2 e in [-125, 8]
    x = np.concatenate([np.linspace(-125.0, 8.0, 3_000_001, dtype=np.float32),
                        np.float32([0.0, -0.5, 0.5, -1.0, 1.0, 7.999, -124.5])])
    got = emulate(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got / want - 1.0)
    assert rel.max() < 8e-5, rel.max()


def test_clamps_instead_of_overflowing_the_exponent():
    got = emulate(np.float32([-200.0, -1e30, -np.inf]))
    assert np.all(got > 0) and np.all(got < 3e-38)
