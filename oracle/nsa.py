"""NSA selection-branch attention forward, float64 CPU oracle.

Source page: "nsa_selection_kernel.py" (openbox-llm).

* Module docstring, "The operation": q ``[B, Hq, T, D]``, k and v
  ``[B, Hkv, T, D]`` with ``Hq = Hkv * G``; ``block_idx [B, Hkv, T, S]`` lists,
  per (batch, kv head, query i), the selected block indices (``block_size``
  tokens each), shared by the G query heads of the group; ``-1`` is padding.
  Query head h uses kv head ``h // G``.  Each query attends to the tokens of its
  selected blocks with keys ``j <= i``, softmax, weighted sum of v; a query with
  no valid selected token outputs 0.
* ``selection_forward_reference`` (the page's ground truth): scale
  ``D**-0.5``; a block listed twice is selected once (a set: one-hot scatter
  followed by ``any``); masked rows are zeroed after the softmax.
* ``_selection_fwd_kernel``: the log-sum-exp ``lse = m + log(l)`` per (query,
  head), natural log, with the finite sentinel ``-1e9`` for an empty row.

Readings taken where the page is silent or inconsistent (listed in the design
notes of the repository):

* ``T % block_size == 0`` is required: the reference clamps tail tokens into
  the last block while the kernel masks them, so the two disagree otherwise.
* An index ``>= T // block_size`` or ``< -1`` is outside the method; the
  oracle raises.
* This oracle gathers per query instead of building the dense T x T score
  matrix (the page notes the dense reference runs out of memory at long
  sequence lengths).  ``nsa_select_dense`` keeps the page's dense formulation
  for tiny inputs, and a CPU test checks the two agree.

TEST INFRASTRUCTURE: see the package docstring for who may import this.
"""

from __future__ import annotations

import numpy as np

LSE_EMPTY = -1.0e9  # lse sentinel of a row with no valid token


def _check(q, k, v, block_idx, block_size):
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    idx = np.asarray(block_idx)
    if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape:
        raise ValueError("q [B,Hq,T,D], k/v [B,Hkv,T,D] expected")
    B, Hq, T, D = q.shape
    Bk, Hkv, Tk, Dk = k.shape
    if (Bk, Tk, Dk) != (B, T, D) or Hq % Hkv != 0:
        raise ValueError("k/v must be [B, Hkv, T, D] with Hq % Hkv == 0")
    if idx.ndim != 4 or idx.shape[:3] != (B, Hkv, T):
        raise ValueError("block_idx must be [B, Hkv, T, S]")
    if T % block_size != 0:
        raise ValueError("T must be a multiple of block_size")
    n_blk = T // block_size
    if idx.size and (idx.min() < -1 or idx.max() >= n_blk):
        raise ValueError("block index out of range")
    return q, k, v, idx


def selected_tokens(sel_row, i: int, block_size: int) -> np.ndarray:
    """Key positions a query at position ``i`` attends to: the tokens of the
    distinct non-negative blocks in ``sel_row`` that satisfy ``j <= i``."""
    blocks = sorted({int(x) for x in sel_row if x >= 0})
    if not blocks:
        return np.zeros(0, dtype=np.int64)
    toks = np.concatenate([np.arange(x * block_size, (x + 1) * block_size) for x in blocks])
    return toks[toks <= i]


def softmax_attend(qg, ks, vs, scale):
    """Softmax attention of the G query rows ``qg [G, D]`` over already
    gathered keys/values ``ks, vs [n, D]``; returns (out [G, D], lse [G]).
    With ``n == 0`` the row is empty: out 0, lse ``-1e9``."""
    qg = np.asarray(qg, dtype=np.float64)
    G, D = qg.shape
    if len(ks) == 0:
        return np.zeros((G, D)), np.full(G, LSE_EMPTY)
    s = (qg @ np.asarray(ks, dtype=np.float64).T) * scale  # [G, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    out = (e @ np.asarray(vs, dtype=np.float64)) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def nsa_select_forward(q, k, v, block_idx, block_size: int):
    """Full NSA selection forward.  Returns ``(out [B,Hq,T,D], lse [B,Hq,T])``."""
    q, k, v, idx = _check(q, k, v, block_idx, block_size)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    scale = float(D) ** -0.5
    out = np.zeros((B, Hq, T, D))
    lse = np.full((B, Hq, T), LSE_EMPTY)
    for b in range(B):
        for g in range(Hkv):
            hs = slice(g * G, (g + 1) * G)
            for i in range(T):
                toks = selected_tokens(idx[b, g, i], i, block_size)
                o, l_ = softmax_attend(q[b, hs, i], k[b, g, toks], v[b, g, toks], scale)
                out[b, hs, i] = o
                lse[b, hs, i] = l_
    return out, lse


def nsa_select_rows(q, k, v, block_idx, block_size: int, rows):
    """NSA selection forward for sampled query groups.

    ``rows`` is a sequence of ``(b, hkv, i)``; returns ``(out [n, G, D],
    lse [n, G])`` for the G query heads ``hkv*G .. hkv*G+G-1`` of each row.
    """
    q, k, v, idx = _check(q, k, v, block_idx, block_size)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    scale = float(D) ** -0.5
    out = np.zeros((len(rows), G, D))
    lse = np.zeros((len(rows), G))
    for n, (b, g, i) in enumerate(rows):
        toks = selected_tokens(idx[b, g, i], i, block_size)
        out[n], lse[n] = softmax_attend(q[b, g * G:(g + 1) * G, i], k[b, g, toks], v[b, g, toks], scale)
    return out, lse


def nsa_select_dense(q, k, v, block_idx, block_size: int) -> np.ndarray:
    """The page's dense ground-truth formulation, for tiny inputs only.

    Builds every score ``q_i.k_j * D**-0.5``, a keep mask = (block of j is
    selected for i, as a set) and (j <= i), fills masked scores with the most
    negative finite float, softmaxes each row and zeroes rows with nothing
    kept, then multiplies by V (``selection_forward_reference``).
    """
    q, k, v, idx = _check(q, k, v, block_idx, block_size)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    n_blk = T // block_size
    scale = float(D) ** -0.5
    kexp = np.repeat(k, G, axis=1)
    vexp = np.repeat(v, G, axis=1)
    s = np.einsum("bhid,bhjd->bhij", q, kexp) * scale
    chosen = np.zeros((B, Hkv, T, n_blk), dtype=bool)
    bb, gg, ii, ss = np.nonzero(idx >= 0)
    chosen[bb, gg, ii, idx[bb, gg, ii, ss]] = True
    blk_of_tok = np.arange(T) // block_size
    keep = chosen[..., blk_of_tok]  # [B,Hkv,T,T]
    keep &= (np.arange(T)[None, :] <= np.arange(T)[:, None])[None, None]
    keep = np.repeat(keep, G, axis=1)
    s = np.where(keep, s, np.finfo(np.float64).min)
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    p = e / e.sum(axis=-1, keepdims=True)
    p = p * keep.any(axis=-1, keepdims=True)
    return p @ vexp


def nsa_pairs(T: int, block_size: int, S: int) -> int:
    """Valid (query, key) pairs per kv group under the synthetic selection
    (current block plus ``min(S-1, c)`` earlier blocks): query i with
    ``c = i // bs`` and ``r = i % bs`` sees ``(r + 1) + bs * min(S-1, c)``."""
    total = 0
    for i in range(T):
        c, r = divmod(i, block_size)
        total += (r + 1) + block_size * min(S - 1, c)
    return total
