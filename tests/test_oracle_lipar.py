"""Pins of the LIPAR pruning / restoration oracle (no GPU).

Fixed by cases with obvious answers: a static clip keeps only frame 0 and
restores every frame from it; tau <= 0 keeps everything; one changed token
keeps exactly its 3 x 3 neighbourhood in that frame (the motion check); a
clip that changes once stays pruned afterwards and restores from the frame
of the change; restoration of kept tokens is the identity.
"""
import numpy as np
import pytest

from oracle import lipar as OL


def _clip(T, H, W, C, seed):
    rng = np.random.default_rng(seed)
    return np.repeat(rng.normal(size=(1, H, W, C)).astype(np.float32), T, axis=0)


def test_static_clip_keeps_frame_zero_only():
    T, H, W, C = 4, 3, 5, 6
    x = _clip(T, H, W, C, 1)
    keep, order, src, n = OL.prune(x.reshape(-1, C), T, H, W, 0.01)
    assert n == H * W and np.array_equal(order, np.arange(H * W))
    assert np.array_equal(src, np.tile(np.arange(H * W), T))


def test_nonpositive_tau_keeps_everything():
    T, H, W, C = 3, 4, 4, 2
    x = _clip(T, H, W, C, 2)
    for tau in (0.0, -1.0):
        keep, order, src, n = OL.prune(x.reshape(-1, C), T, H, W, tau)
        assert keep.all() and n == T * H * W and np.array_equal(src, np.arange(T * H * W))


def test_one_changed_token_keeps_its_neighbourhood():
    T, H, W, C = 3, 6, 7, 4
    x = _clip(T, H, W, C, 3)
    x[1:, 2, 5, 1] += 1.0        # changes at frame 1, then stays
    keep, order, src, n = OL.prune(x.reshape(-1, C), T, H, W, 0.5)
    k = keep.reshape(T, H, W)
    want = np.zeros((H, W), dtype=bool)
    want[1:4, 4:7] = True        # rows 1..3, cols 4..6 (the 3 x 3 around (2, 5))
    assert k[0].all() and np.array_equal(k[1], want) and not k[2].any()
    assert n == H * W + 9
    # frame 2 restores from frame 1 inside the neighbourhood, from frame 0 elsewhere
    F = H * W
    s = src.reshape(T, H, W)
    slot_of = {tok: i for i, tok in enumerate(order)}
    assert s[2, 2, 5] == slot_of[1 * F + 2 * W + 5]
    assert s[2, 0, 0] == slot_of[0]


def test_threshold_is_strict_below_tau():
    T, H, W, C = 2, 1, 1, 3
    x = np.zeros((T, H, W, C), dtype=np.float32)
    x[1, 0, 0, 2] = 0.25
    assert OL.prune(x.reshape(-1, C), T, H, W, 0.25)[3] == 2     # diff == tau: changed
    assert OL.prune(x.reshape(-1, C), T, H, W, 0.2500001)[3] == 1


def test_restore_is_identity_on_kept_tokens():
    rng = np.random.default_rng(5)
    T, H, W, C = 5, 4, 6, 3
    x = rng.normal(size=(T * H * W, C)).astype(np.float32)
    x[H * W:2 * H * W] = x[:H * W]          # frame 1 equals frame 0
    keep, order, src, n = OL.prune(x, T, H, W, 0.1)
    y = rng.normal(size=(n, 8))
    full = OL.restore(y, src)
    assert np.array_equal(full[order], y)
    assert not keep[H * W:2 * H * W].any()  # the repeated frame is pruned


@pytest.mark.parametrize("T,H,W,tau", [(5, 6, 7, 0.5), (4, 1, 9, 0.3), (6, 5, 1, 0.8),
                                       (3, 8, 8, 2.0)])
def test_keep_is_a_3x3_dilation_of_changed(T, H, W, tau):
    # the motion check as a library routine: keep = 3x3 binary dilation of the
    # per-frame changed map, frame 0 always kept
    from scipy.ndimage import binary_dilation
    rng = np.random.default_rng(T * 100 + H * 10 + W)
    x = rng.standard_normal((T, H, W, 4)).astype(np.float32)
    x[1:] = x[:-1] + (rng.random((T - 1, H, W, 1)) < 0.3) * rng.standard_normal(
        (T - 1, H, W, 4)).astype(np.float32)
    keep, order, src, n = OL.prune(x.reshape(T * H * W, 4), T, H, W, tau)
    changed = np.ones((T, H, W), dtype=bool)
    changed[1:] = np.abs(x[1:] - x[:-1]).max(axis=3) >= np.float32(tau)
    want = np.stack([binary_dilation(changed[t], structure=np.ones((3, 3), dtype=bool))
                     for t in range(T)])
    want[0] = True
    assert np.array_equal(keep.reshape(T, H, W), want)
    assert n == int(want.sum()) and np.array_equal(order, np.flatnonzero(want.reshape(-1)))


def test_src_points_to_the_latest_kept_token_at_the_same_position():
    T, H, W = 6, 4, 5
    rng = np.random.default_rng(77)
    x = rng.standard_normal((T, H, W, 3)).astype(np.float32)
    # sparse changes, so tokens stay pruned over several frames
    x = np.repeat(x[:1], T, axis=0)
    for t in range(1, T):
        x[t] = x[t - 1] + (rng.random((H, W, 1)) < 0.04) * 3.0
    keep, order, src, n = OL.prune(x.reshape(T * H * W, 3), T, H, W, 1.0)
    F = H * W
    runs = sum(1 for t in range(2, T) for s in range(F)
               if not keep[t * F + s] and not keep[(t - 1) * F + s])
    assert runs > 0 and 0 < n < T * F  # the case covers pruned runs
    for t in range(T):
        for s in range(F):
            tt = t
            while not keep[tt * F + s]:      # walk back to the latest kept frame
                tt -= 1
            assert order[src[t * F + s]] == tt * F + s
