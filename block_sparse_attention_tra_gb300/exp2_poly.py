"""Minimax polynomial for 2**f on [-1/2, 1/2], used by the threshold-attention
epilogue's FMA-pipe exponential (csrc/tra_math.cuh, ``exp2_fma``).

The epilogue evaluates ``x**p`` as ``exp2(y)`` with ``y = p * log2(x)``.  For
part of the scores it computes ``exp2(y)`` without the MUFU unit, by the
classic range reduction: n = round(y) (an added and subtracted 1.5 * 2**23),
f = y - n in [-1/2, 1/2], ``2**f ~= 1 + f * (c1 + c2 f + ... + cN f**(N-1))``,
and the result's exponent field raised by n with one integer add.  The
coefficients come from the Remez exchange algorithm for the RELATIVE error
with p(0) = 1 exactly (so that y = -127 gives the bit pattern of +0.0), run
here in float64.  With p(0) pinned, the relative error e(f) = (p(f) - 2**f) /
2**f is f (r(f) - g(f)) / 2**f for g(f) = (2**f - 1) / f, r of degree N - 1:
a weighted approximation of g, so the exchange equioscillates e(f) sign(f).

``python -m block_sparse_attention_tra_gb300.exp2_poly [N]`` prints the
coefficients and the float64 and float32-Horner maximum relative errors of
the degree-N fit.
"""

from __future__ import annotations

import sys

import numpy as np

LO, HI = -0.5, 0.5


def _basis(f: np.ndarray, n: int) -> np.ndarray:
    """Columns f, f**2, ..., f**n (the polynomial is 1 at f = 0)."""
    return np.stack([f ** (k + 1) for k in range(n)], axis=-1)


def remez_exp2(n: int, iters: int = 60, grid: int = 200000):
    """Degree-n fit of 2**f on [-1/2, 1/2] with p(0) = 1, minimax in the
    relative error.  Returns (coefficients c1..cn of f..f**n, max rel error)."""
    g = lambda f: 2.0 ** f  # noqa: E731
    k = np.arange(n + 1)
    ref = 0.5 * (LO + HI) - 0.5 * (HI - LO) * np.cos(np.pi * (k + 0.5) / (n + 1))
    ref[ref == 0.0] = 1e-3
    dense = np.linspace(LO, HI, grid)  # an even count: f = 0, where e is 0, is not on the grid
    c = np.zeros(n)
    err = np.inf
    for _ in range(iters):
        # sum_j c_j f_i^j - (-1)^i E sign(f_i) 2^f_i = 2^f_i - 1 at the n + 1 reference points
        alt = ((-1.0) ** np.arange(n + 1)) * np.sign(ref) * g(ref)
        A = np.concatenate([_basis(ref, n), -alt[:, None]], axis=1)
        sol = np.linalg.solve(A, g(ref) - 1.0)
        c = sol[:n]
        e = (1.0 + _basis(dense, n) @ c - g(dense)) / g(dense) * np.sign(dense)
        sgn = np.sign(e)
        sgn[sgn == 0] = 1
        runs = np.flatnonzero(np.diff(sgn)) + 1
        bounds = np.concatenate([[0], runs, [dense.size]])
        ext = [lo + int(np.argmax(np.abs(e[lo:hi]))) for lo, hi in zip(bounds[:-1], bounds[1:])]
        err = float(np.max(np.abs(e)))
        if len(ext) < n + 1:
            break
        best = max(range(len(ext) - n), key=lambda s: min(abs(e[i]) for i in ext[s:s + n + 1]))
        new_ref = dense[ext[best:best + n + 1]]
        if np.allclose(new_ref, ref, atol=1e-12, rtol=0):
            break
        ref = new_ref
    return c, err


def float32_horner_error(c: np.ndarray, grid: int = 2000001) -> float:
    """Max relative error of 1 + f (c1 + ... ) over f in [-1/2, 1/2] with the
    polynomial evaluated in float32 by Horner's rule with fused multiply-adds
    (as the kernel does: r = cN; r = r f + c_k ...; result = r f + 1)."""
    f = np.linspace(LO, HI, grid).astype(np.float32)
    c32 = c.astype(np.float32)
    acc = np.full(f.shape, c32[-1], dtype=np.float32)
    for k in range(len(c32) - 2, -1, -1):
        acc = (acc.astype(np.float64) * f.astype(np.float64) + np.float64(c32[k])).astype(np.float32)
    acc = (acc.astype(np.float64) * f.astype(np.float64) + 1.0).astype(np.float32)
    ref = 2.0 ** f.astype(np.float64)
    return float(np.max(np.abs(acc.astype(np.float64) - ref) / ref))


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    n = int(argv[0]) if argv else 4
    c, err = remez_exp2(n)
    print(f"degree {n}: max |p(f) - 2^f| / 2^f on [-1/2, 1/2] = {err:.3e}"
          f" (float32 Horner {float32_horner_error(c):.3e})")
    print("  {" + ", ".join(f"{x:.9e}f" for x in c) + "}")


if __name__ == "__main__":
    main()
