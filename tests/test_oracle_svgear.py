"""Pins of the SVG-EAR compensation, probe and routing oracle."""
import numpy as np
import pytest

from oracle import attention as A
from oracle import svgear as S


def _qkv(N, d, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((N, d)) * scale, rng.standard_normal((N, d)) * scale,
            rng.standard_normal((N, d)))


def _dense(q, k, v, scale):
    N = k.shape[0]
    o, _ = A.attention_rows(q, k, v, lambda r: np.ones((len(r), N), dtype=bool), scale)
    return o


def test_singleton_key_clusters_are_exact_for_any_selection():
    N, d, Cq = 40, 6, 5
    q, k, v = _qkv(N, d, 1)
    ka = np.random.default_rng(2).permutation(N)          # every key its own cluster
    qa = np.random.default_rng(3).integers(0, Cq, N)
    want = _dense(q, k, v, 0.5)
    for density in (0.0, 0.1, 0.6):
        pr = S.probe(q, k, v, qa, Cq, ka, N, 0.5)
        sel = S.route(pr["err"], pr["nq"], pr["nk"], N, density)
        got = S.compensated_attention(q, k, v, qa, ka, N, sel, 0.5)
        assert np.abs(got - want).max() < 1e-12
        assert np.nanmax(pr["err"]) < 1e-12


def test_full_density_is_exact():
    N, d, Cq, Ck = 60, 5, 4, 7
    q, k, v = _qkv(N, d, 4)
    rng = np.random.default_rng(5)
    qa, ka = rng.integers(0, Cq, N), rng.integers(0, Ck, N)
    pr = S.probe(q, k, v, qa, Cq, ka, Ck, 0.3)
    sel = S.route(pr["err"], pr["nq"], pr["nk"], N, 1.0)
    assert sel[np.ix_(pr["nq"] > 0, pr["nk"] > 0)].all()
    got = S.compensated_attention(q, k, v, qa, ka, Ck, sel, 0.3)
    assert np.abs(got - _dense(q, k, v, 0.3)).max() < 1e-12


def test_zero_density_is_centroid_attention():
    N, d, Cq, Ck = 50, 4, 3, 6
    q, k, v = _qkv(N, d, 6)
    rng = np.random.default_rng(7)
    qa, ka = rng.integers(0, Cq, N), rng.integers(0, Ck, N)
    pr = S.probe(q, k, v, qa, Cq, ka, Ck, 0.8)
    sel = S.route(pr["err"], pr["nq"], pr["nk"], N, 0.0)
    assert not sel.any()
    got = S.compensated_attention(q, k, v, qa, ka, Ck, sel, 0.8)
    assert np.abs(got - S.centroid_attention(q, k, v, ka, Ck, 0.8)).max() < 1e-13


def test_tight_key_clusters_compensate_exactly():
    # keys of one cluster identical (values differ): n_c e^(s q.kc) vc equals
    # the exact sum of the cluster, so compensation is exact and err is 0.
    N, d, Ck = 48, 5, 6
    rng = np.random.default_rng(8)
    ka = rng.integers(0, Ck, N)
    ka[:Ck] = np.arange(Ck)
    kc = rng.standard_normal((Ck, d))
    k = kc[ka]
    q = rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    qa = rng.integers(0, 3, N)
    pr = S.probe(q, k, v, qa, 3, ka, Ck, 0.7)
    assert np.nanmax(np.abs(pr["err"])) < 1e-12
    for density in (0.0, 0.3):
        sel = S.route(pr["err"], pr["nq"], pr["nk"], N, density)
        got = S.compensated_attention(q, k, v, qa, ka, Ck, sel, 0.7)
        assert np.abs(got - _dense(q, k, v, 0.7)).max() < 1e-12


def test_probe_error_is_first_order_output_change():
    # With one query per cluster the proxy is the query itself. Compensating
    # only block (p, c) changes the output by exactly
    # (dE - o dZ) / (Z - dZ); the probe reports |dE - o dZ| / Z.
    N, d, Ck = 30, 4, 5
    q, k, v = _qkv(N, d, 9)
    ka = np.random.default_rng(10).integers(0, Ck, N)
    ka[:Ck] = np.arange(Ck)
    qa = np.arange(N)
    pr = S.probe(q, k, v, qa, N, ka, Ck, 0.6)
    exact = _dense(q, k, v, 0.6)
    for p in (0, 7, 29):
        for c in range(Ck):
            sel = np.ones((N, Ck), dtype=bool)
            sel[p, c] = False
            comp = S.compensated_attention(q, k, v, qa, ka, Ck, sel, 0.6, rows=[p])[0]
            change = np.linalg.norm(exact[p] - comp)
            Z, dZ = pr["Z"][p], pr["dZ"][p, c]
            assert abs(pr["err"][p, c] * Z / (Z - dZ) - change) < 1e-12 * max(1, change)
            # and the direction: exact - compensated = (dE - o dZ) / (Z - dZ)
            r = pr["dE"][p, c] - exact[p] * dZ
            assert np.abs((exact[p] - comp) - r / (Z - dZ)).max() < 1e-12


def test_proxy_error_converges_as_query_clusters_refine():
    # The summary's bound ties the estimate to clustering quality: with finer
    # query clusters the proxy error approaches the per-query error.
    N, d, Ck = 128, 8, 8
    rng = np.random.default_rng(11)
    q = rng.standard_normal((N, d)) * 0.5
    k = rng.standard_normal((N, d)) * 0.5
    v = rng.standard_normal((N, d))
    ka = rng.integers(0, Ck, N)
    truth = S.probe(q, k, v, np.arange(N), N, ka, Ck, 1.0)["err"]    # per query
    order = np.argsort(q[:, 0])                                      # 1-D buckets
    gaps = []
    for Cq in (2, 8, 32, 128):
        qa = np.empty(N, dtype=np.int64)
        qa[order] = np.arange(N) * Cq // N
        err = S.probe(q, k, v, qa, Cq, ka, Ck, 1.0)["err"]
        gaps.append(np.abs(err[qa] - truth).mean())
    assert gaps[-1] < 1e-12
    assert gaps[0] > gaps[1] > gaps[2] > gaps[3]


def test_routing_hand_cases(golden):
    g = golden("routing_cases.txt")
    Cq, Ck, N = map(int, g[2])
    nq = np.array([int(x) for x in g[4]])
    nk = np.array([int(x) for x in g[6]])
    err = np.array([[float(x) for x in g[8]], [float(x) for x in g[9]]])
    for row in g[11:]:
        density = float(row[0])
        want = np.zeros((Cq, Ck), dtype=bool)
        for pc in row[1:]:
            p, c = map(int, pc.split(","))
            want[p, c] = True
        for dt in (np.float64, np.float32):
            got = S.route(err.astype(dt), nq, nk, N, density)
            assert np.array_equal(got, want), (density, dt)


def test_routing_skips_empty_clusters_and_is_a_prefix():
    rng = np.random.default_rng(12)
    Cq, Ck, N = 6, 9, 200
    nq = np.array([40, 0, 60, 30, 50, 20])
    nk = np.array([0, 30, 20, 10, 40, 25, 25, 30, 20])
    err = rng.random((Cq, Ck)).astype(np.float32)
    for density in np.linspace(0, 1, 11):
        sel = S.route(err, nq, nk, N, density)
        assert not sel[1].any() and not sel[:, 0].any()
        cost = (nq[:, None] * nk[None, :])[sel].sum()
        assert cost <= S.budget(density, N)
        # prefix: every unselected valid block ranks below every selected one
        ratio = err / nk.astype(np.float32)[None, :]
        valid = (nq[:, None] > 0) & (nk[None, :] > 0)
        if sel.any() and (valid & ~sel).any():
            assert ratio[sel].min() >= ratio[valid & ~sel].max()


def test_budget_floor():
    assert S.budget(0.15, 32760) == int(np.floor(0.15 * 32760 * 32760))
    assert S.budget(1.0, 7) == 49 and S.budget(0.0, 7) == 0
