"""Linear attention and LinVideo's mixed attention in float64 (TEST INFRASTRUCTURE ONLY).

Sources: LinVideo (gist.science 2510.08318), technical summary sec. 1 (linear
attention lowers the O(n^2) cost of attention to O(n)) and sec. 2 A
(selective transfer: per layer a scalar r in [0, 1] mixes the two kinds,
r = 1 quadratic attention, r = 0 linear attention).

The page names no feature map. Reading: the positive map of Katharopoulos et
al. 2020 ("Transformers are RNNs"), phi(x) = elu(x) + 1 (x + 1 for x > 0,
exp(x) for x <= 0), applied elementwise to q and k as given (no scale), and
the non-causal form (every query sees every key, as in a video DiT's
self-attention). Per batch b, head h and query row i:

    w_ij = phi(q_i) . phi(k_j)                 (> 0)
    lin_i = sum_j w_ij v_j / sum_j w_ij

Mixed attention of a layer with scalar r (reading of "r mixes the two"):

    mix_i = r * att_i + (1 - r) * lin_i

with att_i the block-masked softmax attention of oracle.attention (the
all-ones mask gives the dense quadratic attention of the page).
"""
from __future__ import annotations

import numpy as np

from oracle import attention as OA


def phi(x):
    """elu(x) + 1 in float64."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def linear_rows(q, k, v, rows=None, chunk: int = 256):
    """Linear attention for selected query rows of one (batch, head).

    q, k, v: [N, d]; returns [R, d] float64. Each row is the weighted mean of
    the values with the pairwise weights w_ij above (no factoring of the sum).
    """
    q = np.asarray(q, dtype=np.float64)
    fk = phi(k)
    v = np.asarray(v, dtype=np.float64)
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    out = np.empty((len(rows), v.shape[1]))
    for s in range(0, len(rows), chunk):
        r = rows[s:s + chunk]
        w = phi(q[r]) @ fk.T                      # [R, N] pairwise weights
        out[s:s + len(r)] = (w @ v) / w.sum(axis=1, keepdims=True)
    return out


def linear_attention(q, k, v, rows=None):
    """[B, heads, N, d] inputs; returns [B, heads, R, d] (all rows if rows is None)."""
    B, Hh = q.shape[:2]
    R = q.shape[2] if rows is None else len(rows)
    out = np.empty((B, Hh, R, v.shape[3]))
    for b in range(B):
        for h in range(Hh):
            out[b, h] = linear_rows(q[b, h], k[b, h], v[b, h], rows)
    return out


def mixed_attention(q, k, v, block_mask, block: int, scale: float, r: float, rows=None):
    """r * block-sparse softmax attention + (1 - r) * linear attention."""
    att, _ = OA.block_sparse_attention(q, k, v, block_mask, block, scale, rows=rows)
    lin = linear_attention(q, k, v, rows=rows)
    return r * att + (1.0 - r) * lin
