"""Minimax polynomial for log2(1 + t) on [0, 1), used by the threshold-attention
epilogue's FMA-pipe logarithm (csrc/tra_math.cuh, ``log2_poly``).

The epilogue evaluates ``x**p`` as ``exp2(p * log2(x))``.  For part of the
scores it computes ``log2(x)`` without the MUFU unit: x = 2**e * (1 + t) with
t in [0, 1) (exponent and mantissa fields of the float), and
``log2(1 + t) ~= t * (c1 + c2 t + ... + cN t**(N-1))``.  The coefficients come
from the Remez exchange algorithm (equioscillating absolute error on [0, 1],
with the polynomial forced through 0 at t = 0), run here in float64.

``python -m block_sparse_attention_tra_gb300.log2_poly [N]`` prints the
coefficients and the float64 maximum absolute error of the degree-N fit.
"""

from __future__ import annotations

import sys

import numpy as np


def _basis(t: np.ndarray, n: int) -> np.ndarray:
    """Columns t, t**2, ..., t**n (the polynomial vanishes at t = 0)."""
    return np.stack([t ** (k + 1) for k in range(n)], axis=-1)


def remez_log2(n: int, iters: int = 60, grid: int = 200001):
    """Degree-n minimax fit of log2(1+t) on [0, 1] with p(0) = 0.

    Returns (coefficients c1..cn of t..t**n, max |error|)."""
    f = lambda t: np.log2(1.0 + t)  # noqa: E731
    # initial reference: n + 1 Chebyshev extrema mapped to (0, 1]
    k = np.arange(n + 1)
    ref = 0.5 - 0.5 * np.cos(np.pi * (k + 1) / (n + 1))
    dense = np.linspace(0.0, 1.0, grid)
    c = np.zeros(n)
    err = np.inf
    for _ in range(iters):
        # solve  sum_j c_j t_i^j + (-1)^i E = f(t_i)  at the n + 1 reference points
        A = np.concatenate([_basis(ref, n), ((-1.0) ** np.arange(n + 1))[:, None]], axis=1)
        sol = np.linalg.solve(A, f(ref))
        c = sol[:n]
        e = _basis(dense, n) @ c - f(dense)
        # new reference: the extremum of each sign-alternating run of the error
        sgn = np.sign(e)
        sgn[sgn == 0] = 1
        runs = np.flatnonzero(np.diff(sgn)) + 1
        bounds = np.concatenate([[0], runs, [dense.size]])
        ext = [lo + int(np.argmax(np.abs(e[lo:hi]))) for lo, hi in zip(bounds[:-1], bounds[1:])]
        ext = [i for i in ext if dense[i] > 0.0]  # t = 0 is pinned by the basis
        if len(ext) < n + 1:
            break
        # keep n + 1 consecutive alternating extrema with the largest error
        best = max(range(len(ext) - n), key=lambda s: min(abs(e[i]) for i in ext[s:s + n + 1]))
        new_ref = dense[ext[best:best + n + 1]]
        err = float(np.max(np.abs(e)))
        if np.allclose(new_ref, ref, atol=1e-12, rtol=0):
            break
        ref = new_ref
    return c, err


def mantissa_form(c: np.ndarray) -> np.ndarray:
    """Coefficients a0..an of the same polynomial written in m = 1 + t (the
    kernel evaluates it by Horner's rule directly in the mantissa m in
    [1, 2), which saves the subtraction t = m - 1)."""
    P = np.polynomial.Polynomial(np.concatenate([[0.0], c]))
    return P(np.polynomial.Polynomial([-1.0, 1.0])).coef


def float32_horner_error(a: np.ndarray, grid: int = 2000001) -> float:
    """Max |log2(m) - P(m)| over m in [1, 2) with P evaluated in float32 by
    Horner's rule with fused multiply-adds (as the kernel does)."""
    m = np.linspace(1.0, 2.0, grid, endpoint=False).astype(np.float32)
    a32 = a.astype(np.float32)
    acc = np.full(m.shape, a32[-1], dtype=np.float32)
    for k in range(len(a32) - 2, -1, -1):
        acc = (acc.astype(np.float64) * m.astype(np.float64) + np.float64(a32[k])).astype(np.float32)
    return float(np.max(np.abs(acc.astype(np.float64) - np.log2(m.astype(np.float64)))))


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    n = int(argv[0]) if argv else 5
    c, err = remez_log2(n)
    print(f"degree {n}: max |log2(1+t) - p(t)| on [0,1] = {err:.3e}")
    for j, cj in enumerate(c, 1):
        print(f"  c{j} = {cj:+.9e}")
    a = mantissa_form(c)
    print(f"in m = 1 + t (float32 Horner error {float32_horner_error(a):.3e}):")
    print("  {" + ", ".join(f"{x:.9e}f" for x in a) + "}")


if __name__ == "__main__":
    main()
