"""Pins of the attention-gradient oracle (no GPU).

The gradient oracle is written from the chain rule; it is pinned to things it
does not compute itself:
* central finite differences of the (separately pinned) forward oracle on
  tiny inputs, including a ragged block mask and a query block with no live
  key (its gradient is zero), so a dropped term, a wrong sign, a wrong scale
  or a transposed operand fails;
* one live key per row: the output is that key's value, so dq = dk = 0 and dv
  is the sum of the upstream gradients of the rows that see it;
* invariants of softmax: shifting every key by the same vector leaves every
  row's softmax unchanged, so sum_j dk_j = 0; rows of p sum to 1, so
  sum_j dv_j = sum of g over rows with a live key;
* selecting rows and keys gives the same numbers as the full computation.
"""
import numpy as np
import pytest

from oracle import attention as OA
from oracle import attention_bwd as OB


def _loss(q, k, v, g, bm, block, scale):
    o, _ = OA.block_sparse_attention(q[None, None], k[None, None], v[None, None], bm, block, scale)
    return float((o[0, 0] * g).sum())


def _case(seed, N=10, d=3, block=4):
    rng = np.random.default_rng(seed)
    q, k, v, g = (rng.normal(size=(N, d)) for _ in range(4))
    nb = (N + block - 1) // block
    bm = np.array([[1, 0, 1], [1, 1, 0], [0, 0, 0]], dtype=bool)[:nb, :nb]  # block 2: no live key
    return q, k, v, g, bm, block


@pytest.mark.parametrize("seed", [1, 2])
def test_matches_central_finite_differences(seed):
    q, k, v, g, bm, block = _case(seed)
    scale = 0.7
    dq, dk, dv = OB.block_sparse_attention_grad(q[None, None], k[None, None], v[None, None],
                                                g[None, None], bm, block, scale)
    h = 1e-6
    for name, x, got in (("q", q, dq[0, 0]), ("k", k, dk[0, 0]), ("v", v, dv[0, 0])):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            lp = _loss(**{**args, name: xp}, g=g, bm=bm, block=block, scale=scale)
            lm = _loss(**{**args, name: xm}, g=g, bm=bm, block=block, scale=scale)
            fd[idx] = (lp - lm) / (2 * h)
        assert np.abs(got - fd).max() <= 1e-7, name
    # rows 8, 9 (query block 2) see nothing: zero gradient
    assert not dq[0, 0, 8:].any()


def test_single_live_key_per_row():
    rng = np.random.default_rng(3)
    N, d = 6, 4
    q, k, v, g = (rng.normal(size=(N, d)) for _ in range(4))
    key_of = np.array([0, 0, 2, 5, 5, 5])
    dq, dk, dv = OB.attention_grad(q, k, v, g, lambda r: np.arange(N)[None, :] == key_of[r][:, None],
                                   0.5)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15
    want = np.zeros((N, d))
    for i in range(N):
        want[key_of[i]] += g[i]
    assert np.allclose(dv, want, rtol=0, atol=1e-14)


def test_softmax_invariants():
    rng = np.random.default_rng(4)
    N, d, block = 37, 8, 8
    q, k, v, g = (rng.normal(size=(1, 1, N, d)) for _ in range(4))
    nb = (N + block - 1) // block
    bm = rng.random((nb, nb)) < 0.5
    bm[np.arange(nb), np.arange(nb)] = True
    dq, dk, dv = OB.block_sparse_attention_grad(q, k, v, g, bm, block, 0.3)
    assert np.abs(dk[0, 0].sum(axis=0)).max() < 1e-12
    assert np.allclose(dv[0, 0].sum(axis=0), g[0, 0].sum(axis=0), rtol=0, atol=1e-12)


def test_selected_rows_and_keys_match_full():
    rng = np.random.default_rng(5)
    N, d, block = 50, 4, 16
    q, k, v, g = (rng.normal(size=(1, 2, N, d)) for _ in range(4))
    nb = (N + block - 1) // block
    bm = np.tril(np.ones((nb, nb), dtype=bool))
    full = OB.block_sparse_attention_grad(q, k, v, g, bm, block, 0.5)
    rows, keys = np.array([0, 17, 49]), np.array([3, 33, 48])
    part = OB.block_sparse_attention_grad(q, k, v, g, bm, block, 0.5, rows=rows, keys=keys)
    assert np.allclose(part[0], full[0][:, :, rows], rtol=0, atol=1e-13)
    assert np.allclose(part[1], full[1][:, :, keys], rtol=0, atol=1e-13)
    assert np.allclose(part[2], full[2][:, :, keys], rtol=0, atol=1e-13)
