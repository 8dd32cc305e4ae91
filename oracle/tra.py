"""Threshold rectified attention (TRA) forward, float64 CPU oracle.

Source page: "triton_threshold_attention.py" (snap-research/TDA).

* Module docstring: ``out = (ReLU(Q@K^T - tau))^p @ V`` with the position
  dependent threshold ``tau(i) = beta * sqrt(2 * log(i+1) / d)``.
* ``_threshold_rela_fwd_kernel``: tau per query row from the 0-based row index
  ``i`` as ``(i + 1)``, natural log, ``d`` = head dim; no ``1/sqrt(d)`` factor on
  ``Q@K^T``; causal mask keeps keys ``j <= i``; power branches ``p == 2``,
  ``p == 1`` and a general ``p`` through ``exp(p * log(x))``; the output is the
  unnormalised sum ``sum_j w_ij v_j``.
* ``ThresholdRelaFunction.forward``: q, k, v share the shape ``[B, H, T, D]``.

Readings taken where the page is silent or ambiguous (each listed in the design
notes of the repository):

* Masked (future) pairs contribute nothing.  The page writes 0 into the score
  of a masked pair *before* subtracting tau, which equals "nothing" whenever
  ``beta >= 0`` (then ``ReLU(0 - tau) = 0``); for ``beta < 0`` the page would
  leak ``|tau|^p`` from every future key, which contradicts its own comment
  that a query attends only to positions ``<= i``.
* The general power is the exact ``x**p`` for ``x > 0`` and 0 otherwise; the
  page's ``+1e-10`` inside the log is a guard, not part of the method.
* ``p > 0`` is required (``0**0`` and negative powers are undefined there).

TEST INFRASTRUCTURE: see the package docstring for who may import this.
"""

from __future__ import annotations

import numpy as np


def tau(T: int, beta: float, D: int) -> np.ndarray:
    """Per-row threshold ``tau(i) = beta * sqrt(2 ln(i+1) / D)`` for i = 0..T-1.

    Forward kernel, "Compute tau for each query position": rows are 0-based and
    shifted by one, ``log`` is the natural log, ``D`` is the head dimension.
    """
    i = np.arange(T, dtype=np.float64)
    return float(beta) * np.sqrt(2.0 * np.log(i + 1.0) / float(D))


def relu_power(x: np.ndarray, p: float) -> np.ndarray:
    """``ReLU(x)**p``: ``x**p`` where ``x > 0``, else 0 (forward kernel,
    "Apply threshold" and "Apply power")."""
    if not p > 0:
        raise ValueError("relu power p must be > 0")
    out = np.zeros_like(x, dtype=np.float64)
    pos = x > 0
    out[pos] = np.power(x[pos], float(p))
    return out


def _check(q, k, v):
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one shape [B, H, T, D]")
    return q, k, v


def tra_forward(q, k, v, beta: float, p: float, block: int = 256) -> np.ndarray:
    """Full TRA forward ``out[b,h,i] = sum_{j<=i} ReLU(q_i.k_j - tau(i))^p v_j``.

    Computed row block by row block: for query rows ``i0..i1-1`` the scores
    against keys ``0..i1-1`` come from one BLAS matmul, the causal mask and the
    threshold/power are applied elementwise, and one more matmul multiplies by
    V.  This is the definition written out; the blocking only bounds memory.
    """
    q, k, v = _check(q, k, v)
    B, H, T, D = q.shape
    t = tau(T, beta, D)
    out = np.zeros((B, H, T, D), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for i0 in range(0, T, block):
                i1 = min(T, i0 + block)
                s = q[b, h, i0:i1] @ k[b, h, :i1].T  # [i1-i0, i1]
                x = s - t[i0:i1, None]
                w = relu_power(x, p)
                rows = np.arange(i0, i1)[:, None]
                cols = np.arange(i1)[None, :]
                w[cols > rows] = 0.0  # causal: keys j <= i only
                out[b, h, i0:i1] = w @ v[b, h, :i1]
    return out


def tra_rows(q, k, v, beta: float, p: float, rows) -> np.ndarray:
    """TRA forward for selected output rows only.

    ``rows`` is a sequence of ``(b, h, i)``; returns an array ``[len(rows), D]``
    holding ``out[b, h, i]``.  Used to check full-size launches on sampled rows
    (each row costs O(i*D), independent of the others).
    """
    q, k, v = _check(q, k, v)
    B, H, T, D = q.shape
    t = tau(T, beta, D)
    res = np.zeros((len(rows), D), dtype=np.float64)
    for n, (b, h, i) in enumerate(rows):
        s = k[b, h, : i + 1] @ q[b, h, i]  # [i+1]
        w = relu_power(s - t[i], p)
        res[n] = w @ v[b, h, : i + 1]
    return res


def relu_power_grad(x: np.ndarray, p: float) -> np.ndarray:
    """Derivative of ``ReLU(x)**p``: ``p * x**(p-1)`` where ``x > 0``, else 0.

    The page's backward kernels use the same convention at the kink: the
    derivative is 0 for ``x <= 0`` (p == 1 branch: ``where(qk_thresh > 0, 1,
    0)``; general branch: ``where(qk_relu > 0, ...)``)."""
    if not p > 0:
        raise ValueError("relu power p must be > 0")
    out = np.zeros_like(x, dtype=np.float64)
    pos = x > 0
    out[pos] = float(p) * np.power(x[pos], float(p) - 1.0)
    return out


def tra_backward(q, k, v, dout, beta: float, p: float, block: int = 256):
    """Gradients ``(dq, dk, dv)`` of ``sum(out * dout)`` for the TRA forward.

    Page "triton_threshold_attention.py", ``ThresholdRelaFunction.backward``
    and the kernels ``_threshold_rela_bwd_kernel_dq`` / ``_dkv``: with
    ``x_ij = q_i.k_j - tau(i)`` over the causal pairs ``j <= i``,

        W_ij  = ReLU(x_ij)^p,          dV_j = sum_i W_ij dout_i,
        dA_ij = (dout_i . v_j) * p ReLU(x_ij)^(p-1),
        dQ_i  = sum_j dA_ij k_j,        dK_j = sum_i dA_ij q_i.

    tau does not depend on q or k, and neither beta nor p receives a
    gradient (the page returns None for both).  Masked pairs contribute
    nothing (same reading as the forward).
    """
    q, k, v = _check(q, k, v)
    dout = np.asarray(dout, dtype=np.float64)
    if dout.shape != q.shape:
        raise ValueError("dout must have the shape of q")
    B, H, T, D = q.shape
    t = tau(T, beta, D)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            for i0 in range(0, T, block):
                i1 = min(T, i0 + block)
                x = q[b, h, i0:i1] @ k[b, h, :i1].T - t[i0:i1, None]  # [rows, keys]
                keep = np.arange(i1)[None, :] <= np.arange(i0, i1)[:, None]
                w = np.where(keep, relu_power(x, p), 0.0)
                g = np.where(keep, relu_power_grad(x, p), 0.0)
                da = (dout[b, h, i0:i1] @ v[b, h, :i1].T) * g
                dv[b, h, :i1] += w.T @ dout[b, h, i0:i1]
                dq[b, h, i0:i1] += da @ k[b, h, :i1]
                dk[b, h, :i1] += da.T @ q[b, h, i0:i1]
    return dq, dk, dv


def l2_normalize(x, eps: float = 1e-12) -> np.ndarray:
    """Rows scaled to unit L2 norm along the last axis: ``x / max(||x||, eps)``
    (the page calls ``torch.nn.functional.normalize(x, p=2, dim=-1)``, whose
    default eps is 1e-12)."""
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt((x * x).sum(axis=-1, keepdims=True))
    return x / np.maximum(n, eps)


def tra_diff_forward(q1, q2, k1, k2, v, beta: float, lam: float, p: float, normalize: bool = True,
                     block: int = 256) -> np.ndarray:
    """Threshold differential attention (page "triton_threshold_attention.py",
    ``differential_threshold_rela_triton``):

        out = TRA(q1, k1, v) - clamp(lam, 0, 1) * TRA(q2, k2, v),

    with q1, k1, q2, k2 first L2-normalised row by row when ``normalize``
    (cosine-similarity scores).  Both TRA terms share beta, p and v.
    """
    if normalize:
        q1, q2, k1, k2 = (l2_normalize(a) for a in (q1, q2, k1, k2))
    lam_c = min(max(float(lam), 0.0), 1.0)
    return tra_forward(q1, k1, v, beta, p, block) - lam_c * tra_forward(q2, k2, v, beta, p, block)


def l2_normalize_backward(x, dxn, eps: float = 1e-12) -> np.ndarray:
    """Gradient of ``x -> x / max(||x||, eps)`` (row-wise, last axis) for the
    upstream gradient ``dxn``: with n = ||x|| > eps and xn = x / n,
    ``dx = (dxn - xn (xn . dxn)) / n``; rows with n <= eps (where the map is
    x / eps) give ``dxn / eps``."""
    x = np.asarray(x, dtype=np.float64)
    dxn = np.asarray(dxn, dtype=np.float64)
    n = np.sqrt((x * x).sum(axis=-1, keepdims=True))
    big = n > eps
    xn = x / np.where(big, n, 1.0)
    proj = (xn * dxn).sum(axis=-1, keepdims=True)
    return np.where(big, (dxn - xn * proj) / np.where(big, n, 1.0), dxn / eps)


def tra_diff_backward(q1, q2, k1, k2, v, dout, beta: float, lam: float, p: float, normalize: bool = True):
    """Gradients of ``tra_diff_forward`` (the page's
    ``differential_threshold_rela_triton``, differentiated through its
    normalisation, its two ``ThresholdRelaFunction`` calls and the clamp):

        out = TRA(a1, b1, v) - c TRA(a2, b2, v),  c = clamp(lam, 0, 1),
        a = n(q), b = n(k) (the identity without ``normalize``).

    Returns ``(dq1, dq2, dk1, dk2, dv, dlam)``: each path's (da, db, dv) is
    ``tra_backward`` with the upstream gradient dout and -c dout; dv sums
    both paths; da, db go back through the normalisation; and
    ``dlam = -sum(dout * TRA(a2, b2, v))`` where 0 < lam < 1 (the clamp's
    derivative is 0 outside)."""
    dout = np.asarray(dout, dtype=np.float64)
    ins = [np.asarray(t, dtype=np.float64) for t in (q1, q2, k1, k2)]
    a1, a2, b1, b2 = (l2_normalize(t) for t in ins) if normalize else ins
    c = min(max(float(lam), 0.0), 1.0)
    da1, db1, dv1 = tra_backward(a1, b1, v, dout, beta, p)
    da2, db2, dv2 = tra_backward(a2, b2, v, -c * dout, beta, p)
    dv = dv1 + dv2
    if normalize:
        da1, da2, db1, db2 = (l2_normalize_backward(x, g) for x, g in zip(ins, (da1, da2, db1, db2)))
    dlam = -float((dout * tra_forward(a2, b2, v, beta, p)).sum()) if 0.0 < float(lam) < 1.0 else 0.0
    return da1, da2, db1, db2, dv, dlam


def tra_flops(B: int, H: int, T: int, D: int) -> int:
    """Algorithmic FLOPs of one causal TRA forward: two multiply-adds of length
    D (one for q_i.k_j, one for w_ij v_j) per causally valid pair (i, j<=i)."""
    return 4 * D * B * H * (T * (T + 1) // 2)


def tra_backward_flops(B: int, H: int, T: int, D: int) -> int:
    """Algorithmic FLOPs of one causal TRA backward: per causal pair four
    multiply-adds of length D (dout_i.v_j, dV_j += W dout_i, dQ_i += dA k_j,
    dK_j += dA q_i) plus the recomputed score q_i.k_j."""
    return 10 * D * B * H * (T * (T + 1) // 2)
