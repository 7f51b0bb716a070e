"""Pins of the float64 linear / mixed attention oracle (no GPU).

Each check fixes the oracle against something other than its own formula:
closed-form values of the feature map, a case with a textbook answer
(identical keys give the plain mean of the values), scalar-loop brute force
on tiny inputs, the factored O(N) form the LinVideo page's O(n) claim rests
on (sec. 1), permutation equivariance, and the two ends of the per-layer mix
r (sec. 2 A: r = 1 quadratic, r = 0 linear).
"""
import math

import numpy as np

from oracle import attention as OA
from oracle import linear as OL
from oracle import masks as OM


def test_feature_map_closed_forms():
    x = np.array([0.0, 1.0, 2.5, -1.0, -50.0, 1e-12, -1e-12])
    want = [1.0, 2.0, 3.5, math.exp(-1.0), math.exp(-50.0), 1.0 + 1e-12, math.exp(-1e-12)]
    assert np.allclose(OL.phi(x), want, rtol=1e-15, atol=0.0)
    assert (OL.phi(np.linspace(-30, 30, 1001)) > 0).all()


def test_identical_keys_give_the_mean_value():
    rng = np.random.default_rng(3)
    N, d = 37, 8
    q = rng.normal(size=(N, d))
    k = np.tile(rng.normal(size=(1, d)), (N, 1))
    v = rng.normal(size=(N, d))
    got = OL.linear_rows(q, k, v)
    assert np.allclose(got, np.tile(v.mean(axis=0), (N, 1)), rtol=1e-13, atol=1e-14)


def _brute(q, k, v):
    # scalar loops straight from the definition
    N, d = q.shape
    out = np.zeros((N, v.shape[1]))
    for i in range(N):
        num = [0.0] * v.shape[1]
        den = 0.0
        for j in range(N):
            w = 0.0
            for t in range(d):
                a = q[i, t] + 1.0 if q[i, t] > 0 else math.exp(q[i, t])
                b = k[j, t] + 1.0 if k[j, t] > 0 else math.exp(k[j, t])
                w += a * b
            den += w
            for t in range(v.shape[1]):
                num[t] += w * v[j, t]
        out[i] = [x / den for x in num]
    return out


def test_matches_brute_force_on_tiny_inputs():
    rng = np.random.default_rng(5)
    q, k, v = rng.normal(size=(6, 3)), rng.normal(size=(6, 3)), rng.normal(size=(6, 2))
    assert np.allclose(OL.linear_rows(q, k, v), _brute(q, k, v), rtol=1e-12, atol=1e-13)


def test_factored_form():
    # sum_j (phi(q).phi(k_j)) v_j = phi(q)^T S with S = sum_j phi(k_j) v_j^T, and the
    # denominator phi(q)^T z with z = sum_j phi(k_j)
    rng = np.random.default_rng(7)
    N, d, dv = 50, 5, 4
    q, k, v = rng.normal(size=(N, d)), rng.normal(size=(N, d)), rng.normal(size=(N, dv))
    fk = OL.phi(k)
    S = fk.T @ v
    z = fk.sum(axis=0)
    fq = OL.phi(q)
    want = (fq @ S) / (fq @ z)[:, None]
    assert np.allclose(OL.linear_rows(q, k, v), want, rtol=1e-12, atol=1e-13)


def test_permutation_equivariance():
    rng = np.random.default_rng(9)
    N, d = 40, 6
    q, k, v = rng.normal(size=(N, d)), rng.normal(size=(N, d)), rng.normal(size=(N, d))
    base = OL.linear_rows(q, k, v)
    pk = rng.permutation(N)
    assert np.allclose(OL.linear_rows(q, k[pk], v[pk]), base, rtol=1e-12, atol=1e-13)
    pq = rng.permutation(N)
    assert np.allclose(OL.linear_rows(q[pq], k, v), base[pq], rtol=1e-12, atol=1e-13)


def test_mix_endpoints_and_linearity():
    rng = np.random.default_rng(11)
    T, H, W, d = 3, 4, 5, 8
    N = T * H * W
    q, k, v = (rng.normal(size=(1, 2, N, d)) for _ in range(3))
    p = OM.MaskParams(block=16, w0=3)
    bm = OM.block_mask(OM.RADIAL, T, H, W, p, 0)
    att, _ = OA.block_sparse_attention(q, k, v, bm, 16, 0.25)
    lin = OL.linear_attention(q, k, v)
    assert np.array_equal(OL.mixed_attention(q, k, v, bm, 16, 0.25, 1.0), att)
    assert np.array_equal(OL.mixed_attention(q, k, v, bm, 16, 0.25, 0.0), lin)
    mid = OL.mixed_attention(q, k, v, bm, 16, 0.25, 0.3)
    assert np.allclose(mid, 0.3 * att + 0.7 * lin, rtol=1e-15, atol=1e-15)
    # the output is a convex combination of the values
    assert (np.abs(lin) <= np.abs(v).max() + 1e-12).all()
