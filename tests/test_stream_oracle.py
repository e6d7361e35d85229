"""Pins the oracle of the streaming pipeline (out = alpha * in, binary32).

* the worked example the pages print: N = 2^20, in[i] = (i % 113) * 0.25,
  out = 2 * in, max_error = 0 (tests/golden/scale_by_two_max_error.txt);
* a library routine: numpy's binary32 multiply, element for element;
* special values: zeros, infinities, NaN, subnormals, overflow to infinity.
"""
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scale_by_two_max_error.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if "=" in line:
            k, v = (t.strip() for t in line.split("=", 1))
            vals[k] = v
    return vals


def test_pages_worked_example_max_error_zero():
    g = _golden()
    n = int(g["n"])
    i = np.arange(n, dtype=np.int64)
    x = ((i % 113) * 0.25).astype(np.float32)
    out = oracle.scale_f32(x, float(g["alpha"]))
    max_error = float(np.max(np.abs(out.astype(np.float64) - 2.0 * x.astype(np.float64))))
    assert max_error == float(g["max_error"]) == 0.0


def test_matches_numpy_binary32_multiply():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100003) * 1e3).astype(np.float32)
    for alpha in (2.0, 0.5, -1.5, 1.0 / 3.0, 1e-30):
        a32 = np.float32(alpha)
        ref = x * a32  # numpy: one binary32 rounding per element
        got = oracle.scale_f32(x, alpha)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), alpha


def test_special_values():
    tiny = np.array([1], dtype=np.uint32).view(np.float32)[0]  # smallest subnormal
    x = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, tiny, 3e38, -3e38], dtype=np.float32)
    got = oracle.scale_f32(x, 2.0)
    assert got[0] == 0.0 and not np.signbit(got[0])
    assert got[1] == 0.0 and np.signbit(got[1])
    assert got[2] == np.inf and got[3] == -np.inf and np.isnan(got[4])
    assert got[5:6].view(np.uint32)[0] == 2  # twice the smallest subnormal, exactly
    assert got[6] == np.inf and got[7] == -np.inf
    assert oracle.scale_f32(np.zeros(0, np.float32), 2.0).size == 0
