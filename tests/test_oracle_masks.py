"""Pins of the oracle's mask rules and block pooling."""
import numpy as np
import pytest

from oracle import masks as M


def test_lvsa_tiny_csr_hand_derived(golden):
    g = golden("lvsa_tiny_csr.txt")
    T, H, W, block, local, period, a0, rot, step = map(int, g[1])
    p = M.MaskParams(block=block, local=local, period=period, anchor0=a0, rot_stride=rot)
    rp, col = M.csr(M.LVSA, T, H, W, p, step)
    assert rp.tolist() == [int(x) for x in g[3]]
    assert col.tolist() == [int(x) for x in g[5]]


def test_radial_small_blocks_hand_derived(golden):
    g = golden("radial_small_blocks.txt")
    T, H, W, block, w0 = map(int, g[1])
    want = np.array([[int(x) for x in row] for row in g[3:]], dtype=bool)
    p = M.MaskParams(block=block, w0=w0)
    assert np.array_equal(M.block_mask_literal(M.RADIAL, T, H, W, p), want)
    assert np.array_equal(M.block_mask_segments(M.RADIAL, T, H, W, p), want)


def test_radial_token_pairs_hand_derived(golden):
    g = golden("radial_token_pairs.txt")
    T, H, W, w0 = map(int, g[1])
    F = H * W
    p = M.MaskParams(block=16, w0=w0)
    for ti, si, tj, sj, live in (map(int, r) for r in g[2:]):
        got = bool(M.token_live(M.RADIAL, T, H, W, p, 0, ti * F + si, tj * F + sj))
        assert got == bool(live), (ti, si, tj, sj)


def test_octave_is_bit_length():
    for dt in range(0, 300):
        assert int(M.octave(dt)) == dt.bit_length()


def _radial_pair_count_closed_form(T, F, w0):
    # live token pairs: sum over frame pairs of #{(s_i, s_j): |s_i - s_j| <= w}
    # = F (2w + 1) - w (w + 1) for w < F, F^2 otherwise.
    def f(w):
        return F * F if w >= F - 1 else F * (2 * w + 1) - w * (w + 1)
    total = 0
    for dt in range(T):
        mult = T if dt == 0 else 2 * (T - dt)
        total += mult * f(w0 >> dt.bit_length())
    return total


@pytest.mark.parametrize("T,H,W,w0", [(5, 3, 4, 0), (9, 2, 8, 8), (6, 4, 5, 7), (17, 1, 6, 3)])
def test_radial_token_count_closed_form(T, H, W, w0):
    F = H * W
    p = M.MaskParams(block=8, w0=w0)
    got = int(M.token_mask(M.RADIAL, T, H, W, p).sum())
    assert got == _radial_pair_count_closed_form(T, F, w0 if w0 > 0 else F)


@pytest.mark.parametrize("T,L,P,a0,rho,step", [(7, 1, 0, 0, 1, 0), (11, 2, 3, 1, 2, 1),
                                             (10, 0, 4, 2, 1, 3), (6, 1, 2, 0, 1, 5)])
def test_lvsa_token_count_closed_form(T, L, P, a0, rho, step):
    H, W = 2, 3
    F = H * W
    p = M.MaskParams(block=4, local=L, period=P, anchor0=a0, rot_stride=rho)
    anchors = [t for t in range(T) if ((t - a0 - rho * step) % P == 0 if P > 0 else t == a0)]
    frame_pairs = sum(1 for ti in range(T) for tj in range(T)
                      if abs(ti - tj) <= L or tj in anchors)
    assert int(M.token_mask(M.LVSA, T, H, W, p, step).sum()) == frame_pairs * F * F


def test_lvsa_anchor_rotation():
    p = M.MaskParams(period=3, anchor0=1, rot_stride=2)
    # anchors at step s: t = 1 + 2 s (mod 3)
    assert np.nonzero(M.lvsa_is_anchor(np.arange(9), p, 0))[0].tolist() == [1, 4, 7]
    assert np.nonzero(M.lvsa_is_anchor(np.arange(9), p, 1))[0].tolist() == [0, 3, 6]
    assert np.nonzero(M.lvsa_is_anchor(np.arange(9), p, 2))[0].tolist() == [2, 5, 8]


GRIDS = [(5, 3, 7, 16), (7, 5, 6, 64), (3, 2, 2, 8), (9, 4, 4, 32), (4, 30, 52, 128),
         (2, 5, 5, 64), (3, 1, 1, 2)]


@pytest.mark.parametrize("T,H,W,block", GRIDS)
def test_segment_pooling_equals_token_enumeration(T, H, W, block):
    cases = [(M.RADIAL, M.MaskParams(block=block)), (M.RADIAL, M.MaskParams(block=block, w0=5)),
             (M.LVSA, M.MaskParams(block=block, local=1, period=3, anchor0=1, rot_stride=2)),
             (M.LVSA, M.MaskParams(block=block, local=0, period=0, anchor0=T - 1)),
             (M.DENSE, M.MaskParams(block=block))]
    for kind, p in cases:
        for step in (0, 1):
            lit = M.block_mask_literal(kind, T, H, W, p, step)
            seg = M.block_mask_segments(kind, T, H, W, p, step)
            assert np.array_equal(lit, seg), (kind, p, step)
            # pooling really is "any token pair": recompute from the token mask
            N = T * H * W
            if N > 1200:
                continue
            tm = M.token_mask(kind, T, H, W, p, step)
            nb = M.num_blocks(N, block)
            want = np.zeros((nb, nb), dtype=bool)
            for i in range(N):
                for j in np.nonzero(tm[i])[0]:
                    want[i // block, j // block] = True
            assert np.array_equal(lit, want)


def test_radial_symmetric_and_diagonal():
    p = M.MaskParams(block=64)
    bm = M.block_mask_segments(M.RADIAL, 12, 6, 10, p)
    assert np.array_equal(bm, bm.T)
    assert bm.diagonal().all()
    tm = M.token_mask(M.RADIAL, 4, 3, 5, M.MaskParams(block=4, w0=3))
    assert np.array_equal(tm, tm.T)


def test_lvsa_not_symmetric_anchor_is_key_side():
    bm = M.block_mask_literal(M.LVSA, 4, 8, 8, M.MaskParams(block=64, local=1))
    assert bm[3, 0] and not bm[0, 3]
    assert bm.diagonal().all()


def test_dense_kind_is_all_ones():
    rp, col = M.csr(M.DENSE, 3, 5, 7, M.MaskParams(block=16))
    nb = M.num_blocks(105, 16)
    assert rp.tolist() == [i * nb for i in range(nb + 1)]
    assert col.tolist() == list(range(nb)) * nb


def test_csr_ascending_and_consistent():
    bm = M.block_mask_segments(M.RADIAL, 21, 30, 52, M.MaskParams(block=128))
    rp, col = M.to_csr(bm)
    for r in range(bm.shape[0]):
        seg = col[rp[r]:rp[r + 1]]
        assert (np.diff(seg) > 0).all()
        assert np.array_equal(seg, np.nonzero(bm[r])[0])


def test_workload_counts_cross_check():
    # Counts of the Wan-shaped (21x30x52), LVSA long (126x30x52) and
    # HunyuanVideo 720p (33x45x80) masks, as derived independently when the
    # mask readings were first written down.
    assert M.block_mask_segments(M.RADIAL, 21, 30, 52, M.MaskParams(block=128)).sum() == 29786
    p3 = M.MaskParams(block=128, local=2, period=8, rot_stride=1)
    got = [int(M.block_mask_segments(M.LVSA, 126, 30, 52, p3, s).sum()) for s in range(4)]
    assert got == [402163, 401931, 413643, 401762]
    assert M.block_mask_segments(M.RADIAL, 33, 45, 80, M.MaskParams(block=128)).sum() == 253903


def test_radial_is_n_log_n():
    # With W0 = F each temporal octave adds about F keys per query, so live
    # token pairs / (N * F) grows by a bounded step per doubling of T (log T),
    # while the window W0 >> octave stays >= 1 (here T <= 64 < 2^7, F = 64).
    # Each octave k holds 2^(k-1) frame distances with window F >> k, i.e.
    # about 2 F keys per query per octave; the s_i == s_j pairs add T / F more.
    H, W = 8, 8
    F = H * W
    ratios = []
    for T in (4, 8, 16, 32, 64):
        live = _radial_pair_count_closed_form(T, F, F)
        ratios.append(live / (T * F * F) - T / F)
    steps = np.diff(ratios)
    assert (steps > 1.0).all() and (steps < 2.0).all()
    # dense attention would give a ratio of T (64 at the last point)
    assert ratios[-1] < 10


def test_live_pair_tokens_hand_count_on_a_ragged_grid(golden):
    # The FLOP count behind every TFLOP/s figure: 4 * d * live_pair_tokens.
    g = golden("lvsa_ragged_live_pairs.txt")
    T, H, W, block, local, period, a0 = map(int, g[1])
    want = np.array([[int(x) for x in row] for row in g[3:6]], dtype=bool)
    p = M.MaskParams(block=block, local=local, period=period, anchor0=a0)
    bm = M.block_mask_literal(M.LVSA, T, H, W, p)
    assert np.array_equal(bm, want)
    assert M.live_pair_tokens(bm, block, T * H * W) == int(g[7][0])


@pytest.mark.parametrize("N,block", [(12, 5), (300, 128), (257, 64), (1, 128), (128, 128)])
def test_live_pair_tokens_equals_token_expansion_count(N, block):
    # Independent route: expand the block matrix to its N x N token mask and
    # count the live entries; padding past N never counts.
    rng = np.random.default_rng(N + block)
    nb = M.num_blocks(N, block)
    bm = rng.random((nb, nb)) < 0.4
    assert M.live_pair_tokens(bm, block, N) == int(M.expand_to_tokens(bm, block, N).sum())


def _literal_block_row(kind, T, H, W, p, step, I):
    """Row I of the pooled block mask by literal enumeration of its token pairs."""
    N = T * H * W
    nb = M.num_blocks(N, p.block)
    rows = np.arange(I * p.block, min(N, (I + 1) * p.block))
    live = M.token_live(kind, T, H, W, p, step, rows[:, None], np.arange(N)[None, :])
    padded = np.zeros((len(rows), nb * p.block), dtype=bool)
    padded[:, :N] = live
    return padded.reshape(len(rows), nb, p.block).any(axis=(0, 2))


FULL_GRIDS = [
    # kind, T, H, W, params, steps: the full-size workloads, where the oracle's
    # block_mask takes the frame-run route
    (M.RADIAL, 21, 30, 52, M.MaskParams(block=128), (0,)),
    (M.LVSA, 126, 30, 52, M.MaskParams(block=128, local=2, period=8, rot_stride=1), (0, 1, 2, 3)),
    (M.RADIAL, 33, 45, 80, M.MaskParams(block=128), (0,)),
]


@pytest.mark.parametrize("grid", FULL_GRIDS, ids=["wan_radial", "lvsa_long", "hunyuan_radial"])
def test_frame_run_pooling_matches_literal_rows_at_full_size(grid):
    # Spot check of block_mask_segments against literal token enumeration on
    # whole block rows of the full-size grids: the first, second, a middle, a
    # frame-straddling and the ragged last row.
    kind, T, H, W, p, steps = grid
    N = T * H * W
    nb = M.num_blocks(N, p.block)
    F = H * W
    straddle = next(I for I in range(nb) if (I * p.block) // F != (min(N, (I + 1) * p.block) - 1) // F)
    for step in steps:
        seg = M.block_mask_segments(kind, T, H, W, p, step)
        for I in sorted({0, 1, nb // 2, straddle, nb - 1}):
            lit = _literal_block_row(kind, T, H, W, p, step, I)
            assert np.array_equal(seg[I], lit), (step, I)
