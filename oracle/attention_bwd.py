"""Gradients of masked softmax attention in float64 (TEST INFRASTRUCTURE ONLY).

Radial Attention (hyper.ai news page) adapts pretrained video models to 4x
longer videos by LoRA fine-tuning under its static mask; training runs the
backward pass of the same block-sparse attention. The pages give no formulas
for it, so this is the derivative of the attention definition in
oracle/attention.py by the chain rule. Per batch, head and query row i, with
g_i = dL/do_i the upstream gradient and the masked softmax
p_ij = exp(l_ij - lse_i) (0 where (i, j) is not live):

    dv_j   = sum_i p_ij g_i
    dp_ij  = g_i . v_j
    ds_ij  = p_ij (dp_ij - sum_j' p_ij' dp_ij')      (the softmax Jacobian)
    dq_i   = scale * sum_j ds_ij k_j
    dk_j   = scale * sum_i ds_ij q_i

The inner sum equals g_i . o_i. A row with no live key has o_i = 0 and
contributes nothing.
"""
from __future__ import annotations

import numpy as np


def _row_terms(q, k, v, g, live, scale):
    """p and ds for a chunk of query rows: q, g [r, d]; live [r, N]."""
    logits = np.where(live, scale * (q @ k.T), -np.inf)
    m = logits.max(axis=1)
    has = np.isfinite(m)
    p = np.zeros_like(logits)
    p[has] = np.exp(logits[has] - m[has, None])
    p[has] /= p[has].sum(axis=1, keepdims=True)
    dp = g @ v.T
    delta = (p * dp).sum(axis=1)
    ds = p * (dp - delta[:, None])
    return p, ds


def attention_grad(q, k, v, g, mask_rows, scale: float, rows=None, keys=None, chunk: int = 256):
    """Gradients for one (batch, head).

    q, k, v, g: [N, d] arrays (converted to float64); mask_rows(r) returns the
    boolean token mask [len(r), N]. rows selects the query rows of dq and keys
    the key rows of dk and dv (default: all). Returns (dq [len(rows), d],
    dk [len(keys), d], dv [len(keys), d]) in float64.
    """
    q, k, v, g = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g))
    N = k.shape[0]
    rows = np.arange(N) if rows is None else np.asarray(rows)
    keys = np.arange(N) if keys is None else np.asarray(keys)
    dq = np.zeros((len(rows), q.shape[1]))
    dk = np.zeros((len(keys), k.shape[1]))
    dv = np.zeros((len(keys), v.shape[1]))
    for c0 in range(0, len(rows), chunk):
        r = rows[c0:c0 + chunk]
        _, ds = _row_terms(q[r], k, v, g[r], mask_rows(r), scale)
        dq[c0:c0 + len(r)] = scale * (ds @ k)
    if len(keys) == 0:
        return dq, dk, dv
    # dk and dv need every query row that sees one of the selected keys.
    for c0 in range(0, N, chunk):
        r = np.arange(c0, min(N, c0 + chunk))
        live = mask_rows(r)
        need = live[:, keys].any(axis=1)
        if not need.any():
            continue
        r, live = r[need], live[need]
        p, ds = _row_terms(q[r], k, v, g[r], live, scale)
        dv += p[:, keys].T @ g[r]
        dk += scale * (ds[:, keys].T @ q[r])
    return dq, dk, dv


def block_sparse_attention_grad(q, k, v, g, block_mask, block: int, scale: float, rows=None,
                                keys=None):
    """Gradients of [B, heads, N, d] inputs under a block mask (same for every b, h).

    Token (i, j) is live iff block_mask[i // block, j // block]. Returns
    (dq [B, heads, R, d], dk [B, heads, K, d], dv [B, heads, K, d]) for the
    R selected query rows and K selected key rows.
    """
    B, Hh, N, d = q.shape
    rows_all = np.arange(N) if rows is None else np.asarray(rows)
    keys_all = np.arange(N) if keys is None else np.asarray(keys)

    def mask_rows(r):
        return block_mask[(r // block)[:, None], (np.arange(N) // block)[None, :]]

    dq = np.zeros((B, Hh, len(rows_all), d))
    dk = np.zeros((B, Hh, len(keys_all), d))
    dv = np.zeros((B, Hh, len(keys_all), v.shape[3]))
    for b in range(B):
        for h in range(Hh):
            dq[b, h], dk[b, h], dv[b, h] = attention_grad(q[b, h], k[b, h], v[b, h], g[b, h],
                                                          mask_rows, scale, rows_all, keys_all)
    return dq, dk, dv
