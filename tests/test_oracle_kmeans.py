"""Pins of the float64 Lloyd k-means oracle."""
import warnings

import numpy as np
import pytest

from oracle import kmeans as KM


def _blobs(C, per, d, sep, seed):
    rng = np.random.default_rng(seed)
    centers = rng.standard_normal((C, d)) * sep
    labels = np.repeat(np.arange(C), per)
    x = centers[labels] + rng.standard_normal((C * per, d))
    return x, labels


def test_expanded_distance_matches_definition():
    rng = np.random.default_rng(0)
    x, c = rng.standard_normal((50, 7)), rng.standard_normal((9, 7))
    assert np.abs(KM.sq_distances(x, c) - KM.sq_distances_direct(x, c)).max() < 1e-12


@pytest.mark.parametrize("iters", [1, 3, 50])
def test_matches_sklearn_lloyd(iters):
    from sklearn.cluster import KMeans
    x, _ = _blobs(6, 40, 5, 2.0, seed=1)
    init = np.array([0, 41, 83, 125, 166, 207])
    a, c, n = KM.lloyd(x, init, iters)
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")
        km = KMeans(n_clusters=6, init=x[init], n_init=1, max_iter=iters, tol=0.0,
                    algorithm="lloyd").fit(x)
    # Same centroids after `iters` Lloyd steps. sklearn then relabels every
    # point against those centroids, while the oracle returns the assignment
    # the centroids were computed from; the two agree once Lloyd has converged.
    assert np.abs(c - km.cluster_centers_).max() < 1e-10
    assert np.array_equal(KM.assign(x, c), km.labels_)
    if iters == 50:
        assert np.array_equal(a, km.labels_)
        assert np.array_equal(n, np.bincount(km.labels_, minlength=6))


def test_one_cluster_is_the_mean():
    x = np.random.default_rng(2).standard_normal((30, 4))
    a, c, n = KM.lloyd(x, [7], 3)
    assert (a == 0).all() and n.tolist() == [30]
    assert np.abs(c[0] - x.mean(0)).max() < 1e-14


def test_every_point_its_own_cluster():
    x = np.random.default_rng(3).standard_normal((20, 3))
    init = np.random.default_rng(4).permutation(20)
    a, c, n = KM.lloyd(x, init, 2)
    assert np.array_equal(a[init], np.arange(20))
    assert (n == 1).all() and KM.inertia(x, a, c) == 0.0


def test_ties_go_to_lowest_index():
    x = np.array([[0.0, 0.0]])
    c = np.array([[1.0, 0.0], [0.0, 2.0], [-1.0, 0.0], [0.0, 1.0]])
    # distances 1, 4, 1, 1: clusters 0, 2, 3 tie
    assert KM.assign(x, c).tolist() == [0]
    assert KM.assign(x, c[1:]).tolist() == [1]  # 4, 1, 1 -> index 1 of the slice


def test_empty_cluster_keeps_previous_centroid():
    x = np.array([[0.0], [0.0], [10.0], [11.0]])
    # points 0 and 1 coincide: cluster 1 (init at point 1) ties with cluster 0
    # for every point it could take, so it stays empty and keeps its centroid.
    a, c, n = KM.lloyd(x, [0, 1, 2], 3)
    assert n.tolist() == [2, 0, 2]
    assert c[1, 0] == 0.0
    assert c[2, 0] == 10.5


def test_planted_blobs_recovered():
    x, labels = _blobs(8, 50, 16, 10.0, seed=5)
    init = np.arange(8) * 50 + 3
    a, c, n = KM.lloyd(x, init, 5)
    assert np.array_equal(a, labels)
    assert n.tolist() == [50] * 8


def test_inertia_never_increases():
    x = np.random.default_rng(6).standard_normal((300, 6))
    init = np.random.default_rng(7).choice(300, 12, replace=False)
    prev = np.inf
    for it in range(1, 8):
        a, c, _ = KM.lloyd(x, init, it)
        # inertia of the assignment the centroids were computed from
        val = KM.inertia(x, a, c)
        assert val <= prev + 1e-9
        prev = val


def test_warm_start_from_seed_rows_equals_seeded_lloyd():
    # a warm start from the seed points themselves is the seeded run
    rng = np.random.default_rng(31)
    x = rng.normal(size=(300, 6))
    idx = rng.choice(300, size=9, replace=False)
    for iters in (0, 1, 4):
        a1, c1, n1 = KM.lloyd(x, idx, iters)
        a2, c2, n2 = KM.lloyd_from(x, x[idx], iters)
        assert np.array_equal(a1, a2) and np.array_equal(c1, c2) and np.array_equal(n1, n2)


def test_warm_start_continues_the_iteration():
    # k more iterations from the centroids after m equal m + k iterations
    rng = np.random.default_rng(32)
    x = rng.normal(size=(400, 5))
    idx = rng.choice(400, size=12, replace=False)
    _, c3, _ = KM.lloyd(x, idx, 3)
    a5, c5, n5 = KM.lloyd(x, idx, 5)
    b5, d5, m5 = KM.lloyd_from(x, c3, 2)
    assert np.array_equal(a5, b5) and np.allclose(c5, d5, rtol=0, atol=0) and np.array_equal(n5, m5)
