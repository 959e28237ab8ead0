"""The software exp2 of the row-LSE pass, checked on the CPU against
numpy.exp2 and the fit's error bound: the kernel's constants are read from
its source and its steps (clamp, rounding-constant range reduction, degree-3
polynomial, exponent-field add) are replayed in float32 / uint32."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "query_agnostic_kv_gb300", "csrc", "kvc_recon.cu")


def constants():
    text = open(SRC).read()
    c = {k: np.float32(float(v)) for k, v in re.findall(r"constexpr float (EXP2_C\d|ROUND_MAGIC) = ([0-9.e+-]+)f;", text)}
    clamp = float(re.search(r"x0 = fmaxf\(x0, (-[0-9.]+)f\)", text).group(1))
    return c, np.float32(clamp)


def emulate(x):
    c, clamp = constants()
    x = np.maximum(x.astype(np.float32), clamp)
    t = (x + c["ROUND_MAGIC"]).astype(np.float32)
    n = (t - c["ROUND_MAGIC"]).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = (c["EXP2_C3"] * f + c["EXP2_C2"]).astype(np.float32)
    p = (p * f + c["EXP2_C1"]).astype(np.float32)
    p = (p * f + c["EXP2_C0"]).astype(np.float32)
    bits = (p.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << 23)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def test_relative_error_bound_over_range():
    x = np.linspace(-125.0, 0.0, 2_000_001).astype(np.float32)
    got = emulate(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got / ref - 1.0)
    assert rel.max() < 8e-5, rel.max()
    assert np.all(np.isfinite(got)) and np.all(got > 0)


def test_exact_at_integers_and_monotone_below_clamp():
    x = -np.arange(0, 126, dtype=np.float32)
    got = emulate(x).astype(np.float64)
    assert np.all(np.abs(got / np.exp2(x.astype(np.float64)) - 1) < 8e-5)
    tiny = emulate(np.array([-200.0, -1e30, -np.inf], dtype=np.float32))
    assert np.all(tiny > 0) and np.all(tiny < 1e-37)   # negligible next to a row sum >= 1
