"""LIPAR inter-frame pruning and restoration (TEST INFRASTRUCTURE ONLY).

Source: LIPAR (Latent Inter-frame Pruning with Attention Recovery) summary,
sec. 2 B (pipeline): latent patches whose difference to the same patch of the
previous frame is below a threshold tau are "unchanged"; a motion check with
spatial neighbours guards against pruning slow motion; the unchanged tokens are
removed, attention runs on the shorter sequence, and restoration expands the
result back to full length by duplicating the previous frame's patch.

The page gives no formulas. Readings, per batch b of a latent x[b, t, h, w, :]
(token n = t*H*W + h*W + w):

* changed(t, h, w) = t == 0 or max_c |x[t, h, w, c] - x[t-1, h, w, c]| >= tau
  (the largest channel difference, so the decision is exact in float32);
* keep(t, h, w) = changed at (t, h, w) or at any of its 3 x 3 spatial
  neighbours inside the frame (motion check); frame 0 is always kept;
* compaction: the kept tokens in token order; order[k] = token of slot k,
  n = number of kept tokens;
* restoration: src(t, h, w) = the slot of (t, h, w) if kept, else
  src(t - 1, h, w); out_full[token] = out_compact[src[token]].

M-degree approximation and noise-aware duplication need a RoPE causal model
and its KV cache; they are not part of this reading.
"""
from __future__ import annotations

import numpy as np


def prune(x, T: int, H: int, W: int, tau: float):
    """x: [N, C] latent of one batch (values are used as float32 differences).

    Returns (keep [N] bool, order [n] int64, src [N] int64, n).
    """
    x = np.asarray(x, dtype=np.float32).reshape(T, H, W, -1)
    changed = np.ones((T, H, W), dtype=bool)
    if T > 1:
        diff = np.abs(x[1:] - x[:-1]).max(axis=3)          # exact in float32
        changed[1:] = diff >= np.float32(tau)
    keep = np.zeros((T, H, W), dtype=bool)
    for t in range(T):
        for h in range(H):
            for w in range(W):
                if t == 0:
                    keep[t, h, w] = True
                    continue
                k = False
                for dh in (-1, 0, 1):
                    for dw in (-1, 0, 1):
                        hh, ww = h + dh, w + dw
                        if 0 <= hh < H and 0 <= ww < W and changed[t, hh, ww]:
                            k = True
                keep[t, h, w] = k
    keep = keep.reshape(-1)
    order = np.flatnonzero(keep)
    slot = np.full(keep.shape, -1, dtype=np.int64)
    slot[order] = np.arange(len(order))
    src = np.empty(T * H * W, dtype=np.int64)
    F = H * W
    for t in range(T):
        for s in range(F):
            n = t * F + s
            src[n] = slot[n] if keep[n] else src[n - F]
    return keep, order, src, len(order)


def restore(out_compact, src):
    """out_compact: [n, d]; returns [N, d] with row n = out_compact[src[n]]."""
    return np.asarray(out_compact)[np.asarray(src)]
