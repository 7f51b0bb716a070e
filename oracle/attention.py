"""Masked softmax attention in float64 (TEST INFRASTRUCTURE ONLY).

The pages name block-sparse attention as the operation that video DiTs spend
their time in (LinVideo, gist.science 2510.08318, technical summary sec. 1;
SVG-EAR, gist.science 2603.08982, technical summary sec. 1; LVSA review,
secrett2633 blog, sec. 1) and give no variant of softmax attention, so this is
the textbook definition, per batch b, head h and query row i:

    l_j  = scale * sum_d q[i, d] * k[j, d]    if M[i, j]   else  -inf
    m    = max_j l_j
    p_j  = exp(l_j - m)
    o_i  = sum_j p_j v_j / sum_j p_j
    lse_i = m + log(sum_j p_j)

A row with no live key gives o_i = 0 and lse_i = -inf.
"""
from __future__ import annotations

import numpy as np


def attention_rows(q, k, v, mask_rows, scale: float, rows=None, chunk: int = 256):
    """Attention for selected query rows of one (batch, head).

    q, k, v: [N, d] arrays (converted to float64); mask_rows(rows) returns the
    boolean token mask [len(rows), N]; rows defaults to all N.
    Returns (o [len(rows), d], lse [len(rows)]) in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    N = k.shape[0]
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    o = np.zeros((len(rows), v.shape[1]), dtype=np.float64)
    lse = np.full(len(rows), -np.inf, dtype=np.float64)
    for c0 in range(0, len(rows), chunk):
        r = rows[c0:c0 + chunk]
        live = mask_rows(r)
        assert live.shape == (len(r), N)
        logits = scale * (q[r] @ k.T)
        logits = np.where(live, logits, -np.inf)
        m = logits.max(axis=1)
        has = np.isfinite(m)
        p = np.zeros_like(logits)
        p[has] = np.exp(logits[has] - m[has, None])
        s = p.sum(axis=1)
        o[c0:c0 + len(r)][has] = (p[has] @ v) / s[has, None]
        lse[c0:c0 + len(r)][has] = m[has] + np.log(s[has])
    return o, lse


def block_sparse_attention(q, k, v, block_mask, block: int, scale: float, rows=None):
    """Attention of [B, heads, N, d] inputs under a block mask (same for every b, h).

    Token (i, j) is live iff block_mask[i // block, j // block]. Returns
    (o [B, heads, R, d], lse [B, heads, R]) for the R selected rows.
    """
    B, Hh, N, d = q.shape
    rows_all = np.arange(N) if rows is None else np.asarray(rows)

    def mask_rows(r):
        return block_mask[(r // block)[:, None], (np.arange(N) // block)[None, :]]

    o = np.zeros((B, Hh, len(rows_all), d))
    lse = np.zeros((B, Hh, len(rows_all)))
    for b in range(B):
        for h in range(Hh):
            o[b, h], lse[b, h] = attention_rows(q[b, h], k[b, h], v[b, h], mask_rows, scale, rows_all)
    return o, lse


def sample_rows(N: int, block: int, count: int, seed: int) -> np.ndarray:
    """Sorted distinct query rows: 0, N - 1, the first row of the last block,
    and seeded uniform picks up to `count` rows in total."""
    must = {0, N - 1, ((N - 1) // block) * block}
    rng = np.random.default_rng(seed)
    pool = np.setdiff1d(np.arange(N), np.array(sorted(must)))
    extra = rng.choice(pool, size=max(0, min(count, N) - len(must)), replace=False)
    return np.sort(np.concatenate([np.array(sorted(must)), extra]).astype(np.int64))
