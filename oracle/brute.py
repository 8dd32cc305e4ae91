"""Scalar pure-Python loops of both forwards, for tiny inputs only.

These restate the same definitions as ``oracle.tra`` and ``oracle.nsa`` with
plain Python floats and the ``math`` module -- no numpy, no vectorisation, no
blocking -- so that a vectorisation or indexing slip in the numpy oracle shows
up as a disagreement on small shapes.

Sources: "triton_threshold_attention.py" (module docstring formula,
``_threshold_rela_fwd_kernel``) and "nsa_selection_kernel.py" ("The
operation", ``selection_forward_reference``).

TEST INFRASTRUCTURE: see the package docstring for who may import this.
"""

from __future__ import annotations

import math


def tra_forward(q, k, v, beta, p):
    """q, k, v nested lists [B][H][T][D] of floats -> out [B][H][T][D]."""
    B, H, T, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    out = [[[[0.0] * D for _ in range(T)] for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            for i in range(T):
                t = beta * math.sqrt(2.0 * math.log(i + 1) / D)
                for j in range(i + 1):  # causal: j <= i
                    s = 0.0
                    for d in range(D):
                        s += q[b][h][i][d] * k[b][h][j][d]
                    x = s - t
                    if x <= 0.0:
                        continue
                    w = x ** p
                    for d in range(D):
                        out[b][h][i][d] += w * v[b][h][j][d]
    return out


def tra_backward(q, k, v, dout, beta, p):
    """Scalar loops of the TRA backward; returns (dq, dk, dv) nested lists."""
    B, H, T, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    z = lambda: [[[[0.0] * D for _ in range(T)] for _ in range(H)] for _ in range(B)]  # noqa: E731
    dq, dk, dv = z(), z(), z()
    for b in range(B):
        for h in range(H):
            for i in range(T):
                t = beta * math.sqrt(2.0 * math.log(i + 1) / D)
                for j in range(i + 1):
                    s = sum(q[b][h][i][d] * k[b][h][j][d] for d in range(D))
                    x = s - t
                    if x <= 0.0:
                        continue
                    w = x ** p
                    gw = p * x ** (p - 1.0)
                    dw = sum(dout[b][h][i][d] * v[b][h][j][d] for d in range(D))
                    for d in range(D):
                        dv[b][h][j][d] += w * dout[b][h][i][d]
                        dq[b][h][i][d] += dw * gw * k[b][h][j][d]
                        dk[b][h][j][d] += dw * gw * q[b][h][i][d]
    return dq, dk, dv


def nsa_select_forward(q, k, v, block_idx, block_size):
    """q [B][Hq][T][D], k/v [B][Hkv][T][D], block_idx [B][Hkv][T][S] ->
    (out [B][Hq][T][D], lse [B][Hq][T])."""
    B, Hq, T, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv = len(k[0])
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    out = [[[[0.0] * D for _ in range(T)] for _ in range(Hq)] for _ in range(B)]
    lse = [[[-1.0e9] * T for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i in range(T):
                chosen = set()
                for x in block_idx[b][g][i]:
                    if x >= 0:
                        chosen.add(int(x))
                keys = [j for j in range(i + 1) if j // block_size in chosen]
                if not keys:
                    continue
                scores = []
                for j in keys:
                    s = 0.0
                    for d in range(D):
                        s += q[b][h][i][d] * k[b][g][j][d]
                    scores.append(s * scale)
                m = max(scores)
                es = [math.exp(s - m) for s in scores]
                l = sum(es)
                for e, j in zip(es, keys):
                    for d in range(D):
                        out[b][h][i][d] += e * v[b][g][j][d] / l
                lse[b][h][i] = m + math.log(l)
    return out, lse
