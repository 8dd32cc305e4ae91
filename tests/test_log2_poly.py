"""CPU: the FMA-pipe log2 of the general-power epilogue.

The kernel's coefficients (csrc/tra_math.cuh, LOG2_M) must be the ones the
Remez exchange fit in block_sparse_attention_tra_gb300/log2_poly.py produces,
and the polynomial must meet the error the kernel's accuracy argument uses:
|log2(m) - P(m)| <= 1.6e-5 on [1, 2) when evaluated in float32.  The fit is
also checked against a closed form: an equioscillating error of alternating
sign at n + 2 points (the Chebyshev alternation theorem for the best
approximation).
"""

import os
import re

import numpy as np

from block_sparse_attention_tra_gb300 import log2_poly

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "block_sparse_attention_tra_gb300", "csrc", "tra_math.cuh")


def header_coefficients():
    txt = open(HEADER).read()
    m = re.search(r"LOG2_M\[LOG2_DEG \+ 1\]\s*=\s*\{([^}]*)\}", txt)
    assert m, "LOG2_M not found"
    return np.array([float(x.strip().rstrip("f")) for x in m.group(1).split(",")])


def test_header_coefficients_are_the_remez_fit():
    c, err = log2_poly.remez_log2(5)
    a = log2_poly.mantissa_form(c)
    h = header_coefficients()
    assert h.shape == a.shape
    assert np.allclose(h, a, rtol=2e-8, atol=2e-9), (h, a)
    assert err < 1.5e-5


def test_float32_evaluation_error_bound():
    h = header_coefficients()
    assert log2_poly.float32_horner_error(h) <= 1.6e-5


def test_error_equioscillates():
    # best approximation: n + 2 extrema of equal size and alternating sign
    # (t = 0 is pinned, so the n free coefficients leave n + 1 of them)
    n = 5
    c, err = log2_poly.remez_log2(n)
    t = np.linspace(0.0, 1.0, 400001)
    e = log2_poly._basis(t, n) @ c - np.log2(1.0 + t)
    ext = [i for i in range(1, t.size - 1) if abs(e[i]) >= abs(e[i - 1]) and abs(e[i]) >= abs(e[i + 1])
           and abs(e[i]) > 0.9 * err] + ([t.size - 1] if abs(e[-1]) > 0.9 * err else [])
    signs = np.sign(e[ext])
    assert len(ext) >= n + 1
    assert np.all(signs[1:] != signs[:-1])
    assert np.allclose(np.abs(e[ext]), err, rtol=2e-2)


def test_exact_at_powers_of_two_and_exponent_split():
    # log2 of x = 2^e m: e from the exponent field, P(m) from the mantissa; at
    # m = 1 the polynomial is 0 up to rounding, so powers of two come out exact
    h = header_coefficients()
    assert abs(np.polynomial.polynomial.polyval(1.0, h)) < 1e-6
    x = np.float32([2.0 ** -20, 0.75, 1.5, 3.0, 1000.0])
    bits = x.view(np.uint32)
    e = ((bits >> 23) & 0xFF).astype(np.float64) - 127.0
    m = ((bits & 0x007FFFFF) | 0x3F800000).view(np.float32).astype(np.float64)
    got = e + np.polynomial.polynomial.polyval(m, h)
    assert np.max(np.abs(got - np.log2(x.astype(np.float64)))) < 1.6e-5
