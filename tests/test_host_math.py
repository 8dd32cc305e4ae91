"""CPU checks of host-side arithmetic the kernels rely on.

* The general-power epilogue of the bf16 TRA kernel can evaluate p*log2(x)
  for part of the elements with integer bit operations and a degree-4
  polynomial (constants LOG2_C0..LOG2_C4 in ``csrc/tra_math.cuh``), when
  p >= 1.  Here the same steps are replayed in float32 numpy and checked
  against numpy's log2 over a wide range, including the ReLU zeros whose
  weight must flush to 0.
"""

import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "block_sparse_attention_tra_gb300", "csrc", "tra_math.cuh")


def coefficients():
    txt = open(SRC).read()
    c = [float(re.search(r"LOG2_C%d = ([-+0-9.e]+)f" % k, txt).group(1)) for k in range(5)]
    return np.array(c, dtype=np.float32)


def p_log2_poly2(r, p):
    """float32 replay of p_log2_poly2() in tra_math.cuh (inputs are the ReLU's
    outputs, so r >= 0)."""
    c = coefficients()
    pc = (np.float32(p) * c).astype(np.float32)
    r = np.asarray(r, dtype=np.float32)
    b = r.view(np.uint32)
    m = ((b & np.uint32(0x007FFFFF)) | np.uint32(0x3F800000)).view(np.float32)
    e = ((b >> np.uint32(23)) | np.uint32(0x4B000000)).view(np.float32) - np.float32(8388608.0 + 127.0)
    acc = (pc[4] * m + pc[3]).astype(np.float32)
    acc = (acc * m + pc[2]).astype(np.float32)
    acc = (acc * m + pc[1]).astype(np.float32)
    acc = (acc * m + pc[0]).astype(np.float32)
    return (np.float32(p) * e + acc).astype(np.float32)


def test_log2_polynomial_error_bound():
    r = np.geomspace(1e-37, 1e37, 2_000_001).astype(np.float32)
    for p in (1.5, 3.7, 1.0):
        got = p_log2_poly2(r, p).astype(np.float64)
        want = p * np.log2(r.astype(np.float64))
        # 1.0e-4 from the fit plus float32 rounding of p*e (|p*e| <= ~100)
        tol = p * 1.05e-4 + np.abs(want) * 2 ** -23
        assert np.all(np.abs(got - want) <= tol)


def test_log2_polynomial_relu_zeros_give_zero_weight_for_p_at_least_one():
    """A ReLU zero (x = +0) reads as about -127 p: for p >= 1 its exp2 is below
    the smallest normal float, which ex2.approx.ftz flushes to exactly 0.  (The
    kernels use this path only when p >= 1.)"""
    smallest_normal = np.float64(2.0) ** -126
    for p in (1.0, 1.5, 3.7, 15.0):
        y = p_log2_poly2(np.array([0.0], dtype=np.float32), p).astype(np.float64)
        assert np.all(np.exp2(y) < smallest_normal)
    # Below p = 1 the same bits would give a tiny non-zero weight: excluded.
    y = p_log2_poly2(np.array([0.0], dtype=np.float32), 0.5).astype(np.float64)
    assert np.exp2(y) >= smallest_normal
