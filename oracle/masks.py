"""Static spatiotemporal masks of the oracle (TEST INFRASTRUCTURE ONLY).

Tokens of a latent video of T frames x H x W patches are flattened t-major:
token n has frame t = n // F and in-frame index s = n % F, with F = H * W.

Radial mask (Radial Attention news page, hyper.ai: attention scores decay with
spatial and temporal distance, the static mask keeps mostly nearby tokens and
its window shrinks exponentially with temporal distance, O(n log n) cost).
The page gives no formula; the reading used here is

    live(i, j)  <=>  |s_i - s_j| <= W0 >> octave(|t_i - t_j|)

with octave(0) = 0 and octave(dt) = bit length of dt (1 -> 1, 2..3 -> 2,
4..7 -> 3, ...): the spatial window halves with every octave of temporal
distance, and W0 defaults to F (the whole frame).

LVSA mask (LVSA review, secrett2633 blog, sec. 3 "Method & Key Results" and
Fig. 2: every frame attends a local frame window plus global anchor frames whose
positions rotate with the denoising step). Reading:

    live(i, j)  <=>  |t_i - t_j| <= L   or   t_j is an anchor frame at `step`

with anchors {t : (t - a0 - rho * step) mod P == 0} for a period P > 0, or the
single frame {a0} when P == 0. Anchors are key-side only.

Block pooling (reading of "block-sparse", LVSA review sec. 1): blocks are
[b * block, min(N, (b + 1) * block)); a (query block, key block) pair is live
iff some real token pair in it is live, and a live pair is computed in full.

Two pooling routes are given: ``block_mask_literal`` enumerates token pairs
(small N), ``block_mask_segments`` evaluates the same rule per pair of frame
segments in closed form (any N). Tests check that they agree.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

DENSE, RADIAL, LVSA = 0, 1, 2


@dataclass(frozen=True)
class MaskParams:
    block: int = 128
    w0: int = 0          # radial base window; 0 means F = H * W
    local: int = 1       # LVSA local half-window L (frames)
    period: int = 0      # LVSA anchor period P; 0 means the single anchor a0
    anchor0: int = 0     # LVSA anchor offset a0
    rot_stride: int = 1  # LVSA rotation per denoising step (rho)


def octave(dt):
    """Bit length of non-negative integers (array or int): 0 -> 0, 1 -> 1, 2..3 -> 2."""
    x = np.asarray(dt, dtype=np.int64).copy()
    if (x < 0).any():
        raise ValueError("octave of a negative distance")
    out = np.zeros_like(x)
    while (x > 0).any():
        out += (x > 0)
        x >>= 1
    return out


def radial_window(dt, w0: int):
    """Spatial half-width allowed at temporal distance dt: w0 >> octave(dt)."""
    return np.right_shift(np.int64(w0), octave(dt))


def lvsa_is_anchor(t, p: MaskParams, step: int):
    t = np.asarray(t, dtype=np.int64)
    if p.period > 0:
        return np.mod(t - p.anchor0 - p.rot_stride * step, p.period) == 0
    return t == p.anchor0


def token_live(kind: int, T: int, H: int, W: int, p: MaskParams, step: int, i, j):
    """The token rule for index arrays i (queries) and j (keys), broadcast together."""
    F = H * W
    i = np.asarray(i, dtype=np.int64)
    j = np.asarray(j, dtype=np.int64)
    ti, si = i // F, i % F
    tj, sj = j // F, j % F
    if kind == DENSE:
        return np.ones(np.broadcast(i, j).shape, dtype=bool)
    if kind == RADIAL:
        w0 = p.w0 if p.w0 > 0 else F
        return np.abs(si - sj) <= radial_window(np.abs(ti - tj), w0)
    if kind == LVSA:
        return (np.abs(ti - tj) <= p.local) | lvsa_is_anchor(tj, p, step)
    raise ValueError("unknown mask kind")


def token_mask(kind: int, T: int, H: int, W: int, p: MaskParams, step: int = 0) -> np.ndarray:
    """The N x N token rule itself (no block pooling); small N only."""
    n = np.arange(T * H * W)
    return token_live(kind, T, H, W, p, step, n[:, None], n[None, :])


def num_blocks(N: int, block: int) -> int:
    return (N + block - 1) // block


def block_mask_literal(kind: int, T: int, H: int, W: int, p: MaskParams, step: int = 0) -> np.ndarray:
    """Block pooling by enumerating every real token pair (O(N^2) work)."""
    N = T * H * W
    nb = num_blocks(N, p.block)
    out = np.zeros((nb, nb), dtype=bool)
    cols = np.arange(N)
    for I in range(nb):
        rows = np.arange(I * p.block, min(N, (I + 1) * p.block))
        live = token_live(kind, T, H, W, p, step, rows[:, None], cols[None, :])
        padded = np.zeros((len(rows), nb * p.block), dtype=bool)
        padded[:, :N] = live
        out[I] = padded.reshape(len(rows), nb, p.block).any(axis=(0, 2))
    return out


def frame_segments(start: int, end: int, F: int):
    """Split tokens [start, end) into (frame t, first s, last s) runs."""
    segs = []
    n = start
    while n < end:
        t = n // F
        stop = min(end, (t + 1) * F)
        segs.append((t, n - t * F, stop - 1 - t * F))
        n = stop
    return segs


def _segment_table(N: int, F: int, block: int):
    """Per block, its frame runs as padded arrays (t, lo, hi, valid) of shape [nb, S]."""
    nb = num_blocks(N, block)
    segs = [frame_segments(b * block, min(N, (b + 1) * block), F) for b in range(nb)]
    S = max(len(x) for x in segs)
    t = np.zeros((nb, S), dtype=np.int64)
    lo = np.zeros((nb, S), dtype=np.int64)
    hi = np.zeros((nb, S), dtype=np.int64)
    valid = np.zeros((nb, S), dtype=bool)
    for b, runs in enumerate(segs):
        for r, (tt, a, z) in enumerate(runs):
            t[b, r], lo[b, r], hi[b, r], valid[b, r] = tt, a, z, True
    return t, lo, hi, valid


def block_mask_segments(kind: int, T: int, H: int, W: int, p: MaskParams, step: int = 0) -> np.ndarray:
    """Block pooling by evaluating the rule on pairs of frame runs (any N).

    For a query run (t_i, s in [lo_i, hi_i]) and a key run (t_j, s in
    [lo_j, hi_j]) the smallest |s_i - s_j| is max(0, lo_j - hi_i, lo_i - hi_j),
    so the radial rule holds for some token pair iff that gap is within the
    window of |t_i - t_j|; the LVSA rule depends on the frames alone.
    """
    F = H * W
    N = T * F
    nb = num_blocks(N, p.block)
    t, lo, hi, valid = _segment_table(N, F, p.block)
    out = np.zeros((nb, nb), dtype=bool)
    if kind == DENSE:
        out[:] = True
        return out
    for I in range(nb):
        for a in range(t.shape[1]):
            if not valid[I, a]:
                continue
            ti, lo_i, hi_i = t[I, a], lo[I, a], hi[I, a]
            if kind == RADIAL:
                w0 = p.w0 if p.w0 > 0 else F
                gap = np.maximum(0, np.maximum(lo - hi_i, lo_i - hi))
                live = gap <= radial_window(np.abs(ti - t), w0)
            elif kind == LVSA:
                live = (np.abs(ti - t) <= p.local) | lvsa_is_anchor(t, p, step)
            else:
                raise ValueError("unknown mask kind")
            out[I] |= (live & valid).any(axis=1)
    return out


def block_mask(kind: int, T: int, H: int, W: int, p: MaskParams, step: int = 0) -> np.ndarray:
    """The pooled block mask: literal enumeration up to 8192 tokens, frame runs beyond."""
    if T * H * W <= 8192:
        return block_mask_literal(kind, T, H, W, p, step)
    return block_mask_segments(kind, T, H, W, p, step)


def to_csr(bm: np.ndarray):
    """Row pointers and ascending column indices (int32) of a boolean block matrix."""
    counts = bm.sum(axis=1)
    row_ptr = np.zeros(bm.shape[0] + 1, dtype=np.int64)
    row_ptr[1:] = np.cumsum(counts)
    cols = np.nonzero(bm)[1]            # row-major order: ascending within a row
    return row_ptr.astype(np.int32), cols.astype(np.int32)


def csr(kind: int, T: int, H: int, W: int, p: MaskParams, step: int = 0):
    return to_csr(block_mask(kind, T, H, W, p, step))


def expand_to_tokens(bm: np.ndarray, block: int, N: int, rows=None) -> np.ndarray:
    """Token mask M[i, j] = bm[i // block, j // block] for the given query rows."""
    rows = np.arange(N) if rows is None else np.asarray(rows)
    cols = np.arange(N)
    return bm[(rows // block)[:, None], (cols // block)[None, :]]


def live_pair_tokens(bm: np.ndarray, block: int, N: int) -> int:
    """Sum over live block pairs of |I| * |J| (real tokens only)."""
    nb = bm.shape[0]
    sizes = np.array([min(N, (b + 1) * block) - b * block for b in range(nb)], dtype=np.int64)
    return int((bm * sizes[:, None] * sizes[None, :]).sum())
