"""CPU checks of numerical constants that kernels carry in their source: the
polynomial for log2(1 + t) on [0, 1] that the per-channel-decay chunk kernel
uses in its gates (softplus through one exponential), read from the kernel's
source and evaluated the way the kernel does (fp32, Horner's rule)."""
import os
import re

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
KINTRA = os.path.join(HERE, "..", "continuous_linear_attention_gb300", "csrc", "gdn_kintra.cu")


def _coefficients():
    src = open(KINTRA).read()
    m = re.search(r"kLog2OnePlus\[9\]\s*=\s*\{([^}]*)\}", src)
    assert m, "coefficient table not found"
    vals = [float(v.strip().rstrip("f")) for v in m.group(1).split(",") if v.strip()]
    assert len(vals) == 9
    return np.array(vals, dtype=np.float32)


def _horner_f32(coef, t):
    t = t.astype(np.float32)
    r = np.full_like(t, coef[-1])
    for a in coef[-2::-1]:
        r = (r * t + a).astype(np.float32)  # fmaf rounds once; two roundings here bound it
    return r.astype(np.float64)


def test_log2_one_plus_polynomial_is_accurate_on_the_unit_interval():
    t = np.linspace(0.0, 1.0, 400001)
    err = np.abs(_horner_f32(_coefficients(), t) - np.log2(1.0 + t))
    assert err.max() < 2.5e-7, err.max()
    # the end points, where t = e^{-|x|} sits for |x| = 0 and |x| large
    assert abs(_horner_f32(_coefficients(), np.array([0.0]))[0]) < 1e-7
    assert abs(_horner_f32(_coefficients(), np.array([1.0]))[0] - 1.0) < 2.5e-7


def test_softplus_through_the_polynomial_matches_the_definition():
    """log2(1 + e^x) = max(x, 0) log2 e + p(2^{-|x| log2 e}) against the
    definition over the gate inputs' range (the exponential taken exact here;
    the hardware's adds its own 2^-22 relative error)."""
    coef = _coefficients()
    x = np.linspace(-40.0, 40.0, 200001)
    t = np.exp2(-np.abs(x) * np.log2(np.e)).astype(np.float32)
    got = np.maximum(x, 0.0).astype(np.float32) * np.float32(np.log2(np.e)) + _horner_f32(coef, t)
    want = np.logaddexp(0.0, x) / np.log(2.0)
    # relative to max(1, |value|): fp32 rounding of the large branch plus the polynomial's error
    err = np.abs(got - want) / np.maximum(1.0, np.abs(want))
    assert err.max() < 5e-7, err.max()
