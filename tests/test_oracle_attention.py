"""Pins of the float64 masked-attention oracle."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import masks as M


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_dense_equals_torch_sdpa_float64():
    B, Hh, N, d = 2, 3, 37, 16
    q, k, v = (_rand((B, Hh, N, d), s) for s in (1, 2, 3))
    bm = np.ones((3, 3), dtype=bool)
    scale = 0.3
    o, _ = A.block_sparse_attention(q, k, v, bm, 16, scale)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), scale=scale)
    assert np.abs(o - ref.numpy()).max() < 1e-12


def test_masked_equals_torch_sdpa_with_bool_mask():
    N, d = 45, 8
    q, k, v = (_rand((1, 1, N, d), s) for s in (4, 5, 6))
    p = M.MaskParams(block=8, local=0, period=2)
    bm = M.block_mask_literal(M.LVSA, 5, 3, 3, p)
    o, _ = A.block_sparse_attention(q, k, v, bm, 8, 0.5)
    tm = M.expand_to_tokens(bm, 8, N)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=torch.from_numpy(tm), scale=0.5)
    assert np.abs(o - ref.numpy()).max() < 1e-12


def test_brute_force_python_loops():
    N, d = 6, 3
    q, k, v = _rand((N, d), 7), _rand((N, d), 8), _rand((N, d), 9)
    live = np.array([[(i + j) % 3 != 1 for j in range(N)] for i in range(N)])
    scale = 0.7
    o, lse = A.attention_rows(q, k, v, lambda r: live[r], scale)
    for i in range(N):
        logits = [scale * sum(q[i][c] * k[j][c] for c in range(d)) for j in range(N) if live[i][j]]
        js = [j for j in range(N) if live[i][j]]
        z = sum(math.exp(x) for x in logits)
        for c in range(d):
            want = sum(math.exp(x) * v[j][c] for x, j in zip(logits, js)) / z
            assert abs(o[i][c] - want) < 1e-12
        assert abs(lse[i] - math.log(z)) < 1e-12


def test_rows_sum_to_one():
    N, d = 50, 4
    q, k = _rand((N, d), 10) * 3, _rand((N, d), 11) * 3
    live = _rand((N, N), 12) > 0.3
    live[np.arange(N), np.arange(N)] = True
    o, _ = A.attention_rows(q, k, np.ones((N, 1)), lambda r: live[r], 1.0)
    assert np.abs(o - 1).max() < 1e-13
    # probabilities themselves: v = identity gives the softmax row
    o2, _ = A.attention_rows(q, k, np.eye(N), lambda r: live[r], 1.0)
    assert np.abs(o2.sum(1) - 1).max() < 1e-13
    assert (o2[~live] == 0).all()


def test_permutation_equivariance():
    N, d = 40, 5
    q, k, v = _rand((N, d), 13), _rand((N, d), 14), _rand((N, d), 15)
    live = _rand((N, N), 16) > 0
    live[np.arange(N), np.arange(N)] = True
    perm = np.random.default_rng(17).permutation(N)
    o, lse = A.attention_rows(q, k, v, lambda r: live[r], 0.4)
    lp = live[perm][:, perm]
    op, lsep = A.attention_rows(q[perm], k[perm], v[perm], lambda r: lp[r], 0.4)
    assert np.abs(op - o[perm]).max() < 1e-12
    assert np.abs(lsep - lse[perm]).max() < 1e-12


def test_single_live_key_returns_its_value():
    N, d = 9, 4
    q, k, v = _rand((N, d), 18), _rand((N, d), 19), _rand((N, d), 20)
    target = (np.arange(N) * 4) % N
    live = np.zeros((N, N), dtype=bool)
    live[np.arange(N), target] = True
    o, lse = A.attention_rows(q, k, v, lambda r: live[r], 0.9)
    assert np.abs(o - v[target]).max() < 1e-15
    assert np.abs(lse - 0.9 * (q * k[target]).sum(1)).max() < 1e-13


def test_zero_scale_is_mean_of_live_values():
    N, d = 12, 3
    q, k, v = _rand((N, d), 21), _rand((N, d), 22), _rand((N, d), 23)
    live = _rand((N, N), 24) > 0
    live[:, 0] = True
    o, lse = A.attention_rows(q, k, v, lambda r: live[r], 0.0)
    for i in range(N):
        assert np.abs(o[i] - v[live[i]].mean(0)).max() < 1e-14
        assert abs(lse[i] - math.log(live[i].sum())) < 1e-14


def test_fully_masked_row_is_zero_with_minus_inf_lse():
    N, d = 5, 2
    q, k, v = _rand((N, d), 25), _rand((N, d), 26), _rand((N, d), 27)
    live = np.ones((N, N), dtype=bool)
    live[2] = False
    o, lse = A.attention_rows(q, k, v, lambda r: live[r], 1.0)
    assert (o[2] == 0).all() and lse[2] == -np.inf
    assert np.isfinite(lse[[0, 1, 3, 4]]).all()


def test_block_semantics_compute_whole_live_blocks():
    # A live block pair is computed in full even where the token rule is false.
    T, H, W = 4, 1, 8
    p = M.MaskParams(block=4, w0=2)
    bm = M.block_mask_literal(M.RADIAL, T, H, W, p)
    tm = M.token_mask(M.RADIAL, T, H, W, p)
    ex = M.expand_to_tokens(bm, 4, T * H * W)
    assert (ex >= tm).all() and (ex > tm).any()


def test_sample_rows_includes_edges():
    r = A.sample_rows(1000, 128, 50, seed=3)
    assert len(r) == 50 and len(set(r.tolist())) == 50
    assert {0, 999, 896} <= set(r.tolist())
    assert np.array_equal(r, A.sample_rows(1000, 128, 50, seed=3))
