"""CPU: the FMA-pipe exp2 of the general-power epilogue.

The kernel's coefficients (csrc/tra_math.cuh, EXP2_C) must be the ones the
Remez exchange fit in block_sparse_attention_tra_gb300/exp2_poly.py produces
for degree 4, and meet the error the accuracy argument uses: relative error
<= 3e-6 on [-1/2, 1/2] when evaluated in float32 (against 2^-9, the bf16
rounding of the weight that follows).  The fit is checked against the
alternation theorem, and the kernel's range reduction (round to nearest by an
added and subtracted 1.5 * 2^23, exponent raised by an integer add) is
replayed step for step in float32 against exact powers of two.
"""

import os
import re

import numpy as np

from block_sparse_attention_tra_gb300 import exp2_poly

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "block_sparse_attention_tra_gb300", "csrc", "tra_math.cuh")


def header_coefficients(deg=4):
    txt = open(HEADER).read()
    m = re.search(r"#if BSA_EXP2_DEG == %d\s*__device__ constexpr float EXP2_C\[%d\]\s*=\s*\{([^}]*)\}" % (deg, deg),
                  txt)
    assert m, "EXP2_C not found"
    return np.array([float(x.strip().rstrip("f")) for x in m.group(1).split(",")])


def test_header_coefficients_are_the_remez_fit():
    c, err = exp2_poly.remez_exp2(4)
    h = header_coefficients()
    assert h.shape == c.shape
    assert np.allclose(h, c, rtol=2e-8, atol=2e-9), (h, c)
    assert err < 3e-6
    assert exp2_poly.float32_horner_error(h) <= 3e-6


def test_error_equioscillates():
    # p(0) = 1 is pinned, so the weighted error e(f) sign(f) of the n free
    # coefficients alternates at n + 1 points of equal size
    n = 4
    c, err = exp2_poly.remez_exp2(n)
    f = np.linspace(-0.5, 0.5, 400000)
    e = (1.0 + exp2_poly._basis(f, n) @ c - 2.0 ** f) / 2.0 ** f * np.sign(f)
    ae = np.abs(e)
    ext = [i for i in range(1, f.size - 1) if ae[i] >= ae[i - 1] and ae[i] >= ae[i + 1] and ae[i] > 0.9 * err]
    ext = ([0] if ae[0] > 0.9 * err else []) + ext + ([f.size - 1] if ae[-1] > 0.9 * err else [])
    signs = np.sign(e[ext])
    assert len(ext) >= n + 1
    assert np.all(signs[1:] != signs[:-1])
    assert np.allclose(ae[ext], err, rtol=2e-2)


def kernel_exp2_f32(y):
    """The kernel's steps in float32: clamp, n = round(y) through 1.5 * 2^23,
    f = y - n, Horner with fused multiply-adds, exponent add on the bits."""
    h = header_coefficients().astype(np.float32)
    y = np.minimum(np.maximum(np.float32(y), np.float32(-127.0)), np.float32(128.0)).astype(np.float32)
    magic = np.float32(12582912.0)
    t = (y + magic).astype(np.float32)
    f = (y - (t - magic).astype(np.float32)).astype(np.float32)
    fma = lambda a, b, c: (a.astype(np.float64) * b.astype(np.float64) + np.float64(c)).astype(np.float32)  # noqa: E731
    r = np.full(f.shape, h[-1], dtype=np.float32)
    for k in range(len(h) - 2, -1, -1):
        r = fma(r, f, h[k])
    r = fma(r, f, np.float32(1.0))
    bits = (r.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << 23)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def test_range_reduction_against_exact_powers():
    r = np.random.default_rng(0)
    y = np.concatenate([r.uniform(-126.0, 127.9, 1 << 18), np.arange(-126, 128, dtype=np.float64),
                        np.linspace(-3.0, 3.0, 20001)]).astype(np.float32)
    got = kernel_exp2_f32(y).astype(np.float64)
    ref = np.exp2(y.astype(np.float64))
    assert np.max(np.abs(got - ref) / ref) <= 3.5e-6
    # integers are exact: f = 0 and p(0) = 1
    k = np.arange(-126, 128, dtype=np.float32)
    assert np.array_equal(kernel_exp2_f32(k), np.exp2(k.astype(np.float64)).astype(np.float32))


def test_ends_of_the_range():
    y = np.float32([-np.inf, -1e4, -200.0, -127.0, 128.0, 129.0, 1e4, np.inf])
    w = kernel_exp2_f32(y)
    assert np.all(w[:4] == 0.0) and not np.any(np.signbit(w[:4]))
    assert np.all(np.isposinf(w[4:]))
    # just above -127: a small non-negative subnormal, never a negative or NaN pattern
    s = kernel_exp2_f32(np.float32([-126.99, -126.7, -126.5, -126.3, -126.01]))
    assert np.all(s >= 0.0) and np.all(s < 2.0 ** -125)
