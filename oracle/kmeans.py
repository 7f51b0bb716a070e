"""Lloyd k-means in float64 (TEST INFRASTRUCTURE ONLY).

SVG-EAR (gist.science 2603.08982, technical summary sec. 2, idea 1) groups query
tokens and key tokens by semantic similarity before compensating skipped
blocks with cluster centroids; the page names no algorithm. The reading used
here is plain Lloyd iteration on the raw head vectors with squared Euclidean
distance, per (batch, head):

    centroids <- x[init]                      (init: seeded indices, an input)
    repeat `iters` times:
        assign_i    <- argmin_c ||x_i - c_c||^2   (ties: lowest c)
        centroid_c  <- mean of {x_i : assign_i = c}   (empty: keep previous)
    return assign, centroids, counts

With iters == 0 the result is the assignment to the initial centroids. The
returned centroids are therefore the means of the returned assignment (for
non-empty clusters).
"""
from __future__ import annotations

import numpy as np


def sq_distances_direct(x, c) -> np.ndarray:
    """||x_i - c_c||^2 by the definition (small inputs)."""
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    diff = x[:, None, :] - c[None, :, :]
    return (diff * diff).sum(axis=2)


def sq_distances(x, c) -> np.ndarray:
    """||x_i||^2 - 2 x_i . c_c + ||c_c||^2 in float64.

    The expansion is an algebraic identity of the definition above; its float64
    rounding (about 1e-15 of ||x||^2) is far below any tie tolerance used.
    """
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    return (x * x).sum(1)[:, None] - 2.0 * (x @ c.T) + (c * c).sum(1)[None, :]


def assign(x, c) -> np.ndarray:
    """Index of the nearest centroid; np.argmin returns the first (lowest) minimiser."""
    return np.argmin(sq_distances(x, c), axis=1).astype(np.int64)


def update(x, a, c_prev) -> np.ndarray:
    """Mean of each cluster's members; an empty cluster keeps its previous centroid."""
    x = np.asarray(x, dtype=np.float64)
    C = c_prev.shape[0]
    sums = np.zeros((C, x.shape[1]))
    np.add.at(sums, a, x)
    cnt = np.bincount(a, minlength=C)
    out = np.array(c_prev, dtype=np.float64, copy=True)
    nz = cnt > 0
    out[nz] = sums[nz] / cnt[nz, None]
    return out


def lloyd(x, init_idx, iters: int):
    """One (batch, head): returns (assign [N] int64, centroids [C, d] f64, counts [C] int64)."""
    x = np.asarray(x, dtype=np.float64)
    c = x[np.asarray(init_idx)].copy()
    C = c.shape[0]
    if iters == 0:
        a = assign(x, c)
        return a, c, np.bincount(a, minlength=C)
    for _ in range(iters):
        a = assign(x, c)
        c = update(x, a, c)
    return a, c, np.bincount(a, minlength=C)


def lloyd_from(x, c0, iters: int):
    """Lloyd iterations from given centroids c0 [C, d] (a warm start, e.g. the
    previous denoising step's clusters); otherwise the same steps as lloyd."""
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(c0, dtype=np.float64).copy()
    C = c.shape[0]
    if iters == 0:
        a = assign(x, c)
        return a, c, np.bincount(a, minlength=C)
    for _ in range(iters):
        a = assign(x, c)
        c = update(x, a, c)
    return a, c, np.bincount(a, minlength=C)


def inertia(x, a, c) -> float:
    """Sum of squared distances of points to their assigned centroid."""
    x = np.asarray(x, dtype=np.float64)
    diff = x - np.asarray(c, dtype=np.float64)[np.asarray(a)]
    return float((diff * diff).sum())


def top2_gap(x, c) -> np.ndarray:
    """Per point: second-smallest minus smallest squared distance (tie closeness)."""
    dist = sq_distances(x, c)
    part = np.partition(dist, 1, axis=1)
    return part[:, 1] - part[:, 0]
