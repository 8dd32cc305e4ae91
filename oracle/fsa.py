"""NSA selection forward, block-outer split-K form, float64 CPU oracle.

Source page: "nsa_selection_kernel.py" (openbox-llm), the FSA forward section:
``_selection_fwd_blockouter_kernel`` and ``selection_forward_fsa``.

What the page computes, restated:

* Invert ``block_idx``: for every (batch, kv head, key block j) the list of
  queries that selected j (the page's ``build_block_to_query_csr``, which is
  not printed on the pages).
* For every such (query i, block j) pair and every head g of the group, a
  softmax *partial* over the block's tokens ``t`` with ``t <= i``: the local
  max ``m = max_t s_t``, the denominator ``l = sum_t exp(s_t - m)`` and the
  weighted value sum ``acc = sum_t exp(s_t - m) v_t``, with
  ``s_t = q_i . k_t * D**-0.5``.
* A log-sum-exp combine per (query, head) over its pairs:
  ``M = max_j m_j``, ``w_j = exp(m_j - M)``, ``o = sum_j w_j acc_j / sum_j w_j l_j``,
  ``lse = M + ln(sum_j w_j l_j)``; a row with no pair gives ``o = 0`` and
  the ``-1e9`` sentinel.

Readings (listed in the design notes of the repository):

* The inverted lists hold one pair per distinct non-negative block of a
  query's row whose first token is at or before the query (``j * bs <= i``).
  A pair whose block lies wholly in the future would carry ``l = 0`` and
  weight 0 in the combine (or leave an empty row empty), so leaving it out
  changes nothing; a block listed twice counts once, as in the page's
  ground-truth function.
* The combine is the same math as one softmax over the union of the selected
  causal tokens; ``tests/test_oracle.py`` checks this form against the
  query-outer oracle ``oracle.nsa.nsa_select_forward`` and the dense
  ground-truth formulation.

TEST INFRASTRUCTURE: see the package docstring for who may import this.
"""

from __future__ import annotations

import numpy as np

from .nsa import LSE_EMPTY, _check


def block_query_lists(block_idx, block_size: int):
    """Inverted selection lists: ``{(b, hkv, j): [(i, s), ...]}`` with ``i``
    ascending, ``s`` the first slot of row ``i`` holding ``j``.  Only blocks
    with ``j * block_size <= i`` enter a list."""
    idx = np.asarray(block_idx)
    B, Hkv, T, S = idx.shape
    lists = {}
    for b in range(B):
        for h in range(Hkv):
            for i in range(T):
                seen = set()
                for s in range(S):
                    j = int(idx[b, h, i, s])
                    if j < 0 or j in seen or j * block_size > i:
                        continue
                    seen.add(j)
                    lists.setdefault((b, h, j), []).append((i, s))
    return lists


def fsa_partials(q, k, v, block_idx, block_size: int):
    """Per-(query, block) softmax partials of the block-outer kernel.

    Returns ``{(b, hkv, i, j): (m [G], l [G], acc [G, D])}`` where, over the
    tokens ``t`` of block j with ``t <= i`` and each head g of the group,
    ``m`` is the local max score, ``l = sum exp(s - m)`` and
    ``acc = sum exp(s - m) v_t``; scores are ``q . k * D**-0.5``.
    """
    q, k, v, idx = _check(q, k, v, block_idx, block_size)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    scale = float(D) ** -0.5
    parts = {}
    for (b, h, j), pairs in block_query_lists(idx, block_size).items():
        toks = np.arange(j * block_size, (j + 1) * block_size)
        kb, vb = k[b, h, toks], v[b, h, toks]  # the block's K/V, read once
        for i, _s in pairs:
            qg = q[b, h * G:(h + 1) * G, i]  # [G, D]
            sc = (qg @ kb.T) * scale  # [G, bs]
            keep = toks <= i
            m = sc[:, keep].max(axis=1)
            p = np.where(keep[None, :], np.exp(sc - m[:, None]), 0.0)
            parts[(b, h, i, j)] = (m, p.sum(axis=1), p @ vb)
    return parts


def nsa_select_forward_fsa(q, k, v, block_idx, block_size: int):
    """Block-outer split-K NSA selection forward with the log-sum-exp combine.
    Returns ``(out [B,Hq,T,D], lse [B,Hq,T])``."""
    q, k, v, idx = _check(q, k, v, block_idx, block_size)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    rows = {}
    for (b, h, i, j), part in fsa_partials(q, k, v, idx, block_size).items():
        rows.setdefault((b, h, i), []).append(part)
    out = np.zeros((B, Hq, T, D))
    lse = np.full((B, Hq, T), LSE_EMPTY)
    for (b, h, i), parts in rows.items():
        m = np.stack([p[0] for p in parts])  # [n, G]
        l = np.stack([p[1] for p in parts])  # [n, G]
        acc = np.stack([p[2] for p in parts])  # [n, G, D]
        M = m.max(axis=0)  # [G]
        w = np.exp(m - M[None, :])
        L = (w * l).sum(axis=0)
        hs = slice(h * G, (h + 1) * G)
        out[b, hs, i] = (w[:, :, None] * acc).sum(axis=0) / L[:, None]
        lse[b, hs, i] = M + np.log(L)
    return out, lse
