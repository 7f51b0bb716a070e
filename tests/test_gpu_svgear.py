"""GPU SVG-EAR path (k-means, probe, routing, compensated attention) vs the oracle.

Bars (readings of SVG-EAR, gist.science 2603.08982, technical summary sec. 2):
* k-means: given the same centroids, assignments are bit-exact except points
  whose best and chosen distances are within 1e-4 relative (near-ties, which
  float32 may order either way; counted and bounded); counts equal the
  histogram of the assignment; centroids are the member means (within one
  float32 ulp of the exact mean, checked at 2e-7 relative).
* probe: err within 1e-3 relative (plus a small absolute floor) of the float64
  oracle run on the GPU's clusters.
* routing: (i) bit-exact against the oracle's selection rule applied to the
  GPU's own float32 err; (iii) the selected set equals the oracle's selection
  on its own float64 err, except blocks whose oracle ratio lies within 1e-3
  of the cut ratio (counted and reported).
* Lloyd end to end: the final inertia within 1e-3 relative of the oracle's own
  run from the same initial centroids.
* output: the attention bars (bf16: max-abs 2e-2, mean-abs 2e-3; fp32: 1e-4)
  against the float64 compensated attention with the GPU's selection.
"""
import numpy as np
import pytest
import torch

import synth
from conftest import assert_bf16_close, cached_video_qkv
from oracle import attention as OA
from oracle import kmeans as KM
from oracle import svgear as S

pytestmark = pytest.mark.gpu


def _dev_tensor(x, dev, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev, dtype)


def _assign_ok(x, c, got, rel=1e-4, max_frac=1e-3):
    """got[i] is the oracle's argmin against c, except near-ties (bounded)."""
    dist = KM.sq_distances(x, c)
    want = np.argmin(dist, axis=1)
    bad = np.nonzero(got != want)[0]
    if len(bad):
        i = bad
        gap = dist[i, got[i]] - dist[i, want[i]]
        scale = (x[i] ** 2).sum(1) + (c[want[i]] ** 2).sum(1)
        assert (gap <= rel * scale).all(), ("assignment off beyond a near-tie", int(bad[0]))
        assert len(bad) <= max(1, max_frac * len(got)), ("too many near-ties", len(bad))
    return len(bad)


def _means_ok(x, a, C, cent, count):
    n, means = S.cluster_stats(x, a, C)
    assert np.array_equal(count, n)
    nz = n > 0
    err = np.abs(cent[nz] - means[nz])
    assert (err <= 2e-7 * np.maximum(1.0, np.abs(means[nz]))).all(), float(err.max())


KM_CASES = [
    # B, heads, N, d, C, dtype
    (1, 2, 517, 64, 7, "bf16"),
    (2, 1, 300, 128, 33, "f32"),
    (1, 3, 1000, 128, 100, "bf16"),
    (1, 2, 1500, 128, 300, "bf16"),          # tensor-core path, ragged cluster tile
    (2, 1, 1300, 64, 300, "bf16"),           # the same at head_dim 64: two cluster chunks
]


@pytest.mark.parametrize("case", KM_CASES)
def test_kmeans_iteration_chain(va, dev, case):
    B, Hh, N, d, C, dt = case
    x = synth.iid_qkv(B, Hh, N, d, seed=21, dtype=dt)[0]
    init = synth.init_indices(B, Hh, N, C, seed=22)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    xt = _dev_tensor(x, dev, tdt)
    it = _dev_tensor(init, dev, torch.int32)
    runs = {}
    for iters in (0, 1, 2, 3):
        a, c, n = va.cluster(xt, C, iters, it)
        assert va.device_error() == va.OK
        runs[iters] = (a.cpu().numpy().astype(np.int64), c.cpu().numpy().astype(np.float64),
                       n.cpu().numpy().astype(np.int64))
    for b in range(B):
        for h in range(Hh):
            xs = x[b, h].astype(np.float64)
            # iteration 0: the assignment to the initial centroids x[init]
            a0 = runs[0][0][b, h]
            _assign_ok(xs, xs[init[b, h]], a0)
            assert np.array_equal(runs[0][2][b, h], np.bincount(a0, minlength=C))
            for j in (1, 2, 3):
                a, c, n = (r[b, h] for r in runs[j])
                prev_c = xs[init[b, h]] if j == 1 else runs[j - 1][1][b, h]
                _assign_ok(xs, prev_c, a)
                _means_ok(xs, a, C, c, n)


def test_kmeans_recovers_planted_blobs(va, dev):
    rng = np.random.default_rng(5)
    C, per, d = 16, 40, 64
    centers = rng.standard_normal((C, d)) * 6.0
    labels = np.repeat(np.arange(C), per)
    x = (centers[labels] + rng.standard_normal((C * per, d))).astype(np.float32)
    init = np.arange(C, dtype=np.int32) * per + 3        # one seed point per blob
    a, c, n = va.cluster(_dev_tensor(x[None, None], dev, torch.float32), C, 5,
                         _dev_tensor(init[None, None], dev, torch.int32))
    assert np.array_equal(a.cpu().numpy()[0, 0], labels)
    assert (n.cpu().numpy()[0, 0] == per).all()
    want = np.stack([x[labels == k].astype(np.float64).mean(0) for k in range(C)])
    assert np.abs(c.cpu().numpy()[0, 0] - want).max() < 1e-5


def test_kmeans_rejects_bad_arguments(va, dev):
    x = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16, device=dev)
    init = torch.arange(8, dtype=torch.int32, device=dev).view(1, 1, 8)
    with pytest.raises(va.VAError) as e:
        va.cluster(x, 8, -1, init)
    assert e.value.status == va.ERR_INVALID
    x96 = torch.zeros((1, 1, 64, 96), dtype=torch.bfloat16, device=dev)
    with pytest.raises(va.VAError) as e:
        va.cluster(x96, 8, 1, init)
    assert e.value.status == va.ERR_UNSUPPORTED
    bad = torch.full((1, 1, 8), 64, dtype=torch.int32, device=dev)   # index == N
    va.cluster(x, 8, 1, bad)
    assert va.device_error() == va.ERR_DEVICE
    assert va.device_error() == va.OK


def _route_case(va, dev, q, k, v, qa, ka, Cq, Ck, density, scale, dt):
    B, Hh, N, d = q.shape
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    qt, kt, vt = (_dev_tensor(x, dev, tdt) for x in (q, k, v))
    err = torch.empty((B, Hh, Cq, Ck), dtype=torch.float32, device=dev)
    sel = torch.empty((B, Hh, Cq, Ck), dtype=torch.uint8, device=dev)
    out, _, _ = va.compensate_route(qt, kt, vt, _dev_tensor(qa, dev, torch.int32), Cq,
                                    _dev_tensor(ka, dev, torch.int32), Ck, density,
                                    scale=scale, err=err, sel=sel)
    assert va.device_error() == va.OK
    return out.float().cpu().numpy(), err.cpu().numpy(), sel.cpu().numpy().astype(bool)


def _check_err(got, want, rel=1e-3):
    finite = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), finite)
    floor = 1e-6 * max(1e-30, np.abs(want[finite]).max())
    diff = np.abs(got[finite] - want[finite])
    assert (diff <= rel * np.abs(want[finite]) + floor).all(), float((diff / (np.abs(want[finite]) + floor)).max())


ROUTE_CASES = [
    # N, d, Cq, Ck, density, dtype, empty clusters
    (331, 128, 5, 17, 0.2, "bf16", True),
    (331, 64, 6, 13, 0.0, "f32", False),
    (400, 128, 4, 11, 1.0, "f32", True),
    (700, 128, 9, 40, 0.15, "bf16", False),
    # tensor-core probe: a ragged second proxy tile, empty clusters, many splits
    (2500, 128, 130, 150, 0.1, "bf16", True),
    # clusters longer than a 64-key tile
    (1500, 128, 3, 7, 0.3, "bf16", False),
    # head_dim 64 on the tensor-core compensated attention
    (331, 64, 5, 17, 0.2, "bf16", True),
    (2500, 64, 130, 150, 0.1, "bf16", True),
    (1500, 64, 3, 7, 0.3, "bf16", False),
]


@pytest.mark.parametrize("case", ROUTE_CASES)
def test_compensate_route_small(va, dev, case):
    N, d, Cq, Ck, density, dt, empty = case
    B, Hh = 1, 2
    T = 1
    q, k, v = synth.video_qkv(B, Hh, T, 1, N, d, seed=31, dtype=dt)
    rng = np.random.default_rng(32)
    qa = rng.integers(0, Cq - (1 if empty else 0), (B, Hh, N)).astype(np.int32)
    ka = rng.integers(0, Ck - (2 if empty else 0), (B, Hh, N)).astype(np.int32)
    scale = 1.0 / np.sqrt(d)
    out, err, sel = _route_case(va, dev, q, k, v, qa, ka, Cq, Ck, density, scale, dt)
    for b in range(B):
        for h in range(Hh):
            pr = S.probe(q[b, h], k[b, h], v[b, h], qa[b, h], Cq, ka[b, h], Ck, scale)
            _check_err(err[b, h], pr["err"])
            want_sel = S.route(err[b, h], pr["nq"], pr["nk"], N, density)
            assert np.array_equal(sel[b, h], want_sel)
            _near_cut_agreement(sel[b, h], pr["err"], pr["nq"], pr["nk"], N, density)
            want = S.compensated_attention(q[b, h], k[b, h], v[b, h], qa[b, h], ka[b, h], Ck,
                                           sel[b, h], scale)
            if dt == "bf16":
                assert_bf16_close(out[b, h], want)
            else:
                assert np.abs(out[b, h] - want).max() <= 1e-4


def test_compensate_route_extremes_match_closed_forms(va, dev):
    # density 1: exact dense attention; singleton key clusters: exact for any density.
    N, d = 256, 64
    q, k, v = synth.iid_qkv(1, 1, N, d, seed=41)
    scale = 0.125
    rng = np.random.default_rng(42)
    qa = rng.integers(0, 4, (1, 1, N)).astype(np.int32)
    dense, _ = OA.attention_rows(q[0, 0], k[0, 0], v[0, 0],
                                 lambda r: np.ones((len(r), N), dtype=bool), scale)
    ka = rng.integers(0, 8, (1, 1, N)).astype(np.int32)
    out, _, sel = _route_case(va, dev, q, k, v, qa, ka, 4, 8, 1.0, scale, "f32")
    assert sel.all()
    assert np.abs(out[0, 0] - dense).max() <= 1e-4
    ka1 = rng.permutation(N).astype(np.int32).reshape(1, 1, N)
    out, err, _ = _route_case(va, dev, q, k, v, qa, ka1, 4, N, 0.05, scale, "f32")
    assert np.abs(out[0, 0] - dense).max() <= 1e-4
    assert np.nanmax(err) < 1e-5


@pytest.mark.parametrize("d", [128, 64])
def test_compensate_route_running_max_rises_every_tile(va, dev, d):
    # Keys' logits grow with their index and key clusters are index ranges, so
    # each of the four centroid tiles (128 clusters) raises the row max by
    # about 51 (log2 units), past the rescale threshold: the bf16 softmax takes
    # its max pass and rescales O on those entries, then meets exact tiles
    # below the max it has reached.
    N, Cq, Ck = 2048, 4, 512
    rng = np.random.default_rng(44)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    q = 8.0 * u[None, :] + 0.05 * rng.standard_normal((N, d))
    k = (200.0 * np.arange(N) / N)[:, None] * u[None, :] + 0.05 * rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    q, k, v = (torch.from_numpy(x.reshape(1, 1, N, d).astype(np.float32)).bfloat16().float()
               .numpy() for x in (q, k, v))
    qa = rng.integers(0, Cq, (1, 1, N)).astype(np.int32)
    ka = (np.arange(N) * Ck // N).astype(np.int32).reshape(1, 1, N)
    scale = 1.0 / np.sqrt(d)
    out, err, sel = _route_case(va, dev, q, k, v, qa, ka, Cq, Ck, 0.3, scale, "bf16")
    assert np.isfinite(out).all()
    nq = np.bincount(qa[0, 0], minlength=Cq)
    nk = np.bincount(ka[0, 0], minlength=Ck)
    assert np.array_equal(sel[0, 0], S.route(err[0, 0], nq, nk, N, 0.3))
    want = S.compensated_attention(q[0, 0], k[0, 0], v[0, 0], qa[0, 0], ka[0, 0], Ck, sel[0, 0],
                                   scale)
    assert_bf16_close(out[0, 0], want)


def _near_cut_agreement(sel_gpu, err_oracle, nq, nk, N, density, rel=1e-3):
    """Routing reading (iii): the GPU's selected set against the oracle's
    selection on its own float64 errors. Blocks whose oracle ratio lies within
    `rel` of the cut ratio may go either way; every other block must agree.
    Returns (blocks near the cut, disagreements)."""
    want = S.route(err_oracle, nq, nk, N, density)
    valid = (nq[:, None] > 0) & (nk[None, :] > 0)
    ratio = np.where(valid, err_oracle / np.maximum(nk, 1)[None, :], -np.inf)
    cut = ratio[want].min() if want.any() else np.inf
    near = valid & (np.abs(ratio - cut) <= rel * abs(cut))
    diff = sel_gpu != want
    assert not (diff & ~near).any(), ("selection differs away from the cut",
                                      np.argwhere(diff & ~near)[:5].tolist())
    return int(near.sum()), int(diff.sum())


def test_svgear_full_size(va, dev):
    # SVG-EAR-style workload: B=1, 12 heads, 21x30x52 = 32,760 tokens, d=128,
    # bf16; k-means with 256 query and 1,024 key clusters (10 iterations,
    # seeded init); routing at 15% density with centroid compensation. Every
    # head is checked: the last k-means step given the GPU's previous
    # centroids, the end-to-end Lloyd inertia against the oracle's own run from
    # the same seed indices, the probe errors, the routing against the oracle's
    # selection on its own float64 errors, and 512 sampled output rows.
    import oracle_jobs
    T, H, W, Hh, d, Cq, Ck, density = 21, 30, 52, 12, 128, 256, 1024, 0.15
    N = T * H * W
    scale = 1.0 / np.sqrt(d)
    q, k, v = cached_video_qkv(1, Hh, T, H, W, d, seed=1238)
    qinit_h = synth.init_indices(1, Hh, N, Cq, seed=1238, tensor=synth.INIT)
    kinit_h = synth.init_indices(1, Hh, N, Ck, seed=1238, tensor=synth.INIT + 1)
    pool = oracle_jobs.spawn_pool(2 * Hh)
    try:
        lloyd_q = [pool.apply_async(oracle_jobs.lloyd_run, (q[0, h], qinit_h[0, h], 10))
                   for h in range(Hh)]
        lloyd_k = [pool.apply_async(oracle_jobs.lloyd_run, (k[0, h], kinit_h[0, h], 10))
                   for h in range(Hh)]
        qt, kt, vt = (_dev_tensor(x, dev, torch.bfloat16) for x in (q, k, v))
        qinit, kinit = _dev_tensor(qinit_h, dev, torch.int32), _dev_tensor(kinit_h, dev, torch.int32)
        qa9, qc9, _ = va.cluster(qt, Cq, 9, qinit)
        qa, qc, qn = va.cluster(qt, Cq, 10, qinit)
        ka9, kc9, _ = va.cluster(kt, Ck, 9, kinit)
        ka, kc, kn = va.cluster(kt, Ck, 10, kinit)
        assert va.device_error() == va.OK
        qa, ka = qa.cpu().numpy(), ka.cpu().numpy()
        qc9, kc9, qc, kc = (t.cpu().numpy().astype(np.float64) for t in (qc9, kc9, qc, kc))
        qn, kn = qn.cpu().numpy(), kn.cpu().numpy()
        probes = [pool.apply_async(oracle_jobs.probe_err, (q[0, h], k[0, h], v[0, h], qa[0, h],
                                                           Cq, ka[0, h], Ck, scale))
                  for h in range(Hh)]
        near_ties = 0
        for h in range(Hh):
            qs, ks = q[0, h].astype(np.float64), k[0, h].astype(np.float64)
            near_ties += _assign_ok(qs, qc9[0, h], qa[0, h].astype(np.int64))
            near_ties += _assign_ok(ks, kc9[0, h], ka[0, h].astype(np.int64))
            _means_ok(qs, qa[0, h], Cq, qc[0, h], qn[0, h])
            _means_ok(ks, ka[0, h], Ck, kc[0, h], kn[0, h])
        for x, a, c, runs in ((q, qa, qc, lloyd_q), (k, ka, kc, lloyd_k)):
            for h in range(Hh):
                got = KM.inertia(x[0, h], a[0, h], c[0, h])
                _, want = runs[h].get()
                assert abs(got - want) <= 1e-3 * want, (h, got, want)
        err = torch.empty((1, Hh, Cq, Ck), dtype=torch.float32, device=dev)
        sel = torch.empty((1, Hh, Cq, Ck), dtype=torch.uint8, device=dev)
        out, _, _ = va.compensate_route(qt, kt, vt, _dev_tensor(qa, dev, torch.int32), Cq,
                                        _dev_tensor(ka, dev, torch.int32), Ck, density, err=err,
                                        sel=sel)
        assert va.device_error() == va.OK
        err, sel, out = err.cpu().numpy(), sel.cpu().numpy().astype(bool), out.float().cpu().numpy()
        rows = OA.sample_rows(N, 128, 512, seed=9)
        near_cut = flips = 0
        for h in range(Hh):
            nq, _ = S.cluster_stats(q[0, h], qa[0, h], Cq)
            nk, _ = S.cluster_stats(k[0, h], ka[0, h], Ck)
            # (i) the selection rule, bit-exact on the GPU's own float32 errors
            assert np.array_equal(sel[0, h], S.route(err[0, h], nq, nk, N, density))
            cost = (nq[:, None] * nk[None, :])[sel[0, h]].sum()
            assert cost <= S.budget(density, N)
            # (ii) the errors against the oracle's float64 probe
            err_o = probes[h].get()
            _check_err(err[0, h], err_o)
            # (iii) the selected set against the oracle's selection on its own errors
            n_near, n_diff = _near_cut_agreement(sel[0, h], err_o, nq, nk, N, density)
            near_cut += n_near
            flips += n_diff
            want = S.compensated_attention(q[0, h], k[0, h], v[0, h], qa[0, h], ka[0, h], Ck,
                                           sel[0, h], scale, rows=rows)
            assert_bf16_close(out[0, h][rows], want)
        print("svgear full size: k-means near-ties %d; routing: %d blocks within 1e-3 of the "
              "cut, %d selected differently (all of them near the cut)"
              % (near_ties, near_cut, flips))
    finally:
        pool.terminate()
        pool.join()


@pytest.mark.parametrize("B,Hh,N,d,C,dt", [(1, 2, 1500, 128, 300, "bf16"),  # tensor cores, 2 chunks
                                            (2, 1, 517, 64, 7, "f32"),      # FMA path
                                            (1, 1, 700, 128, 40, "bf16")])  # one ragged chunk
def test_kmeans_warm_start_chain_vs_oracle(va, dev, B, Hh, N, d, C, dt):
    # va_cluster_from against oracle/kmeans.lloyd_from, from centroids that
    # are not seed rows (a previous step's clusters, modelled as seed rows
    # moved by N(0, 0.1^2) noise): every iteration's assignment is the oracle's
    # argmin given the same centroids (near-ties bounded), the centroids are
    # the member means, and after 3 iterations the inertia is within 1e-3 of
    # the oracle's own lloyd_from run from the same start.
    x = synth.iid_qkv(B, Hh, N, d, seed=61, dtype=dt)[0]
    init = synth.init_indices(B, Hh, N, C, seed=62)
    rng = np.random.default_rng(63)
    c0 = np.stack([np.stack([x[b, h][init[b, h]] for h in range(Hh)]) for b in range(B)])
    c0 = (c0 + 0.1 * rng.standard_normal(c0.shape)).astype(np.float32)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    xt = _dev_tensor(x, dev, tdt)
    c0t = _dev_tensor(c0, dev, torch.float32)
    runs = {}
    for iters in (0, 1, 2, 3):
        a, c, n = va.cluster_from(xt, c0t, iters)
        assert va.device_error() == va.OK
        runs[iters] = (a.cpu().numpy().astype(np.int64), c.cpu().numpy().astype(np.float64),
                       n.cpu().numpy().astype(np.int64))
    for b in range(B):
        for h in range(Hh):
            xs = x[b, h].astype(np.float64)
            c0s = c0[b, h].astype(np.float64)
            a0 = runs[0][0][b, h]
            _assign_ok(xs, c0s, a0)
            assert np.array_equal(runs[0][2][b, h], np.bincount(a0, minlength=C))
            for j in (1, 2, 3):
                a, c, n = (r[b, h] for r in runs[j])
                prev_c = c0s if j == 1 else runs[j - 1][1][b, h]
                _assign_ok(xs, prev_c, a)
                _means_ok(xs, a, C, c, n)
            a_o, c_o, _ = KM.lloyd_from(xs, c0s, 3)
            got = KM.inertia(xs, runs[3][0][b, h], runs[3][1][b, h])
            want = KM.inertia(xs, a_o, c_o)
            assert abs(got - want) <= 1e-3 * want, (got, want)


@pytest.mark.parametrize("B,Hh,N,d,C", [(1, 2, 1500, 128, 300),   # tensor-core path, 2 chunks
                                         (2, 1, 517, 64, 7)])     # FMA path
def test_kmeans_warm_start_from_seed_rows_equals_seeded(va, dev, B, Hh, N, d, C):
    # warm start (reuse across denoising steps): starting from the float copies
    # of the seed rows is the seeded run, bit for bit
    x = torch.from_numpy(synth.iid_qkv(B, Hh, N, d, seed=51)[0]).to(dev, torch.bfloat16)
    init = torch.from_numpy(synth.init_indices(B, Hh, N, C, seed=52)).to(dev)
    c0 = torch.stack([torch.stack([x[b, h, init[b, h].long()].float() for h in range(Hh)])
                      for b in range(B)]).contiguous()
    for iters in (0, 3):
        a1, c1, n1 = va.cluster(x, C, iters, init)
        a2, c2, n2 = va.cluster_from(x, c0, iters)
        torch.cuda.synchronize()
        assert va.device_error() == va.OK
        assert torch.equal(a1, a2) and torch.equal(c1, c2) and torch.equal(n1, n2)


def test_kmeans_warm_start_continues_the_iteration(va, dev):
    # 4 iterations from the centroids after 6 give the result after 10
    q, _, _ = cached_video_qkv(1, 2, 8, 32, 32, 128, seed=53)
    x = torch.from_numpy(q).to(dev, torch.bfloat16)
    N, C = x.shape[2], 256
    init = torch.from_numpy(synth.init_indices(1, 2, N, C, seed=54)).to(dev)
    a10, c10, n10 = va.cluster(x, C, 10, init)
    _, c6, _ = va.cluster(x, C, 6, init)
    a, c, n = va.cluster_from(x, c6, 4, centroid=c6)     # in place
    torch.cuda.synchronize()
    assert va.device_error() == va.OK
    assert torch.equal(a, a10) and torch.equal(c, c10) and torch.equal(n, n10)


@pytest.mark.parametrize("d,dt", [(128, "bf16"), (64, "bf16"), (128, "f32")])
def test_repeated_calls_are_bit_identical(va, dev, d, dt):
    """Member lists hold each cluster's tokens in ascending order (no atomic
    slot order), so every sum over them, and with them the errors, the
    routing, the output and the fp32 k-means, repeats bit for bit."""
    B, Hh, N, Cq, Ck = 1, 3, 3000, 40, 150
    q, k, v = synth.video_qkv(B, Hh, 1, 1, N, d, seed=41, dtype=dt)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    qt, kt, vt = (_dev_tensor(x, dev, tdt) for x in (q, k, v))
    rng = np.random.default_rng(42)
    qa = _dev_tensor(rng.integers(0, Cq, (B, Hh, N)).astype(np.int32), dev, torch.int32)
    ka = _dev_tensor(rng.integers(0, Ck, (B, Hh, N)).astype(np.int32), dev, torch.int32)
    runs = []
    for _ in range(3):
        err = torch.empty((B, Hh, Cq, Ck), dtype=torch.float32, device=dev)
        sel = torch.empty((B, Hh, Cq, Ck), dtype=torch.uint8, device=dev)
        out, _, _ = va.compensate_route(qt, kt, vt, qa, Cq, ka, Ck, 0.15, err=err, sel=sel)
        runs.append((out.clone(), err.clone(), sel.clone()))
    assert va.device_error() == va.OK
    for o, e, s in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(e, runs[0][1])
        assert torch.equal(s, runs[0][2])
    init = _dev_tensor(synth.init_indices(B, Hh, N, Cq, seed=43), dev, torch.int32)
    res = []
    for _ in range(2):
        a = torch.empty((B, Hh, N), dtype=torch.int32, device=dev)
        c = torch.empty((B, Hh, Cq, d), dtype=torch.float32, device=dev)
        n = torch.empty((B, Hh, Cq), dtype=torch.int32, device=dev)
        va.cluster(qt, Cq, 4, init, a, c, n)
        res.append((a, c, n))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
    assert torch.equal(res[0][2], res[1][2])
