"""Fit the polynomial used by the tcgen05 TRA epilogue for log2 on [1, 2).

The epilogue splits x = 2^e * m (m in [1, 2)) with integer bit operations
and approximates log2(m) by a degree-4 polynomial in m, fitted here by least
squares on Chebyshev nodes of [1, 2] (a near-minimax fit).  Run this script
to regenerate the constants LOG2_C0..LOG2_C4 of ``tra_math.cuh``; it prints the header and
the maximum absolute error of the fit in float64 and when evaluated in
float32 Horner form.
"""

import numpy as np

DEG = 4


def fit(deg=DEG, n=4000):
    x = np.cos(np.pi * (np.arange(n) + 0.5) / n) * 0.5 + 1.5
    V = np.vander(x, deg + 1, increasing=True)
    c, *_ = np.linalg.lstsq(V, np.log2(x), rcond=None)
    return c


def eval_f32(c, m):
    m = m.astype(np.float32)
    acc = np.float32(c[-1])
    for ck in c[-2::-1]:
        acc = (acc * m + np.float32(ck)).astype(np.float32)
    return acc


if __name__ == "__main__":
    c = fit()
    mt = np.linspace(1.0, 2.0, 1_000_001)
    e64 = np.abs(np.polyval(c[::-1], mt) - np.log2(mt)).max()
    e32 = np.abs(eval_f32(c, mt).astype(np.float64) - np.log2(mt)).max()
    print("// log2(m) ~= sum_k LOG2_POLY[k] * m^k on [1, 2); max |err| %.2e (f64), %.2e (f32 Horner)" % (e64, e32))
    print("constexpr float " + ", ".join("LOG2_C%d = %.9ef" % (k, v) for k, v in enumerate(c)) + ";")
