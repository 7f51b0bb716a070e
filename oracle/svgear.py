"""Centroid compensation, error probe and error-aware routing (TEST INFRASTRUCTURE ONLY).

Source: SVG-EAR (gist.science 2603.08982), technical summary sec. 2:
idea 1 (parameter-free linear compensation: the contribution of a skipped
block is approximated through the cluster centroids), idea 2 (error-aware
routing: estimate each block's compensation error with a light probe that uses
query-cluster centroids as proxies, cost O(C_q N_k d) instead of O(N_q N_k d),
streamed without storing logits; under a density budget compute exactly the
blocks with the highest error-to-cost ratio and compensate the rest).

The page gives no formulas. Readings used here (one batch, one head; scale s):

* A block is a (query cluster p, key cluster c) pair; n_p, n_c are the
  cluster sizes; kc_c, vc_c, qc_p are member means (float64).
* Compensated term of key cluster c for query i: the n_c keys of c are
  replaced by one virtual key kc_c with logit bias ln n_c and value vc_c, i.e.
  numerator n_c exp(s q_i.kc_c) vc_c and denominator n_c exp(s q_i.kc_c).
* Probe with proxy q~ = qc_p, logits l_j = s q~.k_j, m_p = max_j l_j:
      Z_p = sum_j e^(l_j - m_p),  O_p = sum_j e^(l_j - m_p) v_j / Z_p
      dE  = sum_{j in c} e^(l_j - m_p) v_j - n_c e^(s q~.kc_c - m_p) vc_c
      dZ  = sum_{j in c} e^(l_j - m_p)     - n_c e^(s q~.kc_c - m_p)
      err(p, c) = || dE - O_p dZ ||_2 / Z_p
  which is the first-order change of the proxy's normalised output when block
  (p, c) is compensated instead of computed.
* cost(p, c) = n_p n_c token pairs; ratio = n_p err / cost = err / n_c.
* Routing: order blocks by ratio descending (ties: p ascending, then c
  ascending), keep the longest prefix whose cumulative cost is at most
  floor(density * N * N). Blocks with an empty cluster are never selected.
* Output for query i in cluster p with selected set S(p): exact terms for keys
  in selected clusters, compensated terms for the other non-empty clusters,
  one softmax over both (shared max).
"""
from __future__ import annotations

import math

import numpy as np


def cluster_stats(x, a, C: int):
    """(counts [C] int64, means [C, d] float64); an empty cluster's mean is 0."""
    x = np.asarray(x, dtype=np.float64)
    a = np.asarray(a, dtype=np.int64)
    n = np.bincount(a, minlength=C).astype(np.int64)
    sums = np.zeros((C, x.shape[1]))
    np.add.at(sums, a, x)
    means = np.zeros_like(sums)
    means[n > 0] = sums[n > 0] / n[n > 0, None]
    return n, means


def probe(q, k, v, qa, Cq: int, ka, Ck: int, scale: float):
    """err [Cq, Ck] float64 (NaN where a cluster is empty) plus the probe terms.

    Returns a dict with err, Z [Cq], O [Cq, d], dE [Cq, Ck, d], dZ [Cq, Ck].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, qc = cluster_stats(q, qa, Cq)
    nk, kc = cluster_stats(k, ka, Ck)
    _, vc = cluster_stats(v, ka, Ck)
    ka = np.asarray(ka, dtype=np.int64)
    d = v.shape[1]
    err = np.full((Cq, Ck), np.nan)
    Z = np.zeros(Cq)
    O = np.zeros((Cq, d))
    dE = np.zeros((Cq, Ck, d))
    dZ = np.zeros((Cq, Ck))
    for p in range(Cq):
        if nq[p] == 0:
            continue
        l = scale * (k @ qc[p])                      # [N] logits of the proxy
        m = l.max()
        e = np.exp(l - m)
        Z[p] = e.sum()
        O[p] = (e @ v) / Z[p]
        E_c = np.zeros((Ck, d))                      # exact block numerators
        np.add.at(E_c, ka, e[:, None] * v)
        Z_c = np.bincount(ka, weights=e, minlength=Ck)
        lc = scale * (kc @ qc[p])
        w = nk * np.exp(lc - m)                      # compensated weights
        dE[p] = E_c - w[:, None] * vc
        dZ[p] = Z_c - w
        r = dE[p] - O[p][None, :] * dZ[p][:, None]
        e_pc = np.sqrt((r * r).sum(axis=1)) / Z[p]
        err[p] = np.where(nk > 0, e_pc, np.nan)
    return {"err": err, "Z": Z, "O": O, "dE": dE, "dZ": dZ, "nq": nq, "nk": nk}


def budget(density: float, N: int) -> int:
    """floor(density * N * N) in IEEE double."""
    return int(math.floor(float(density) * float(N) * float(N)))


def route(err, nq, nk, N: int, density: float) -> np.ndarray:
    """Selected blocks as a boolean [Cq, Ck] matrix.

    ratio = err / n_c in err's own dtype (so float32 errors give float32
    ratios, rounded as IEEE division does).
    """
    err = np.asarray(err)
    nq = np.asarray(nq, dtype=np.int64)
    nk = np.asarray(nk, dtype=np.int64)
    Cq, Ck = err.shape
    P, Cidx = np.meshgrid(np.arange(Cq), np.arange(Ck), indexing="ij")
    valid = (nq[:, None] > 0) & (nk[None, :] > 0)
    ratio = err / nk.astype(err.dtype)[None, :] if err.dtype == np.float32 else err / nk[None, :]
    p_v, c_v, r_v = P[valid], Cidx[valid], ratio[valid]
    cost = nq[p_v] * nk[c_v]
    # np.lexsort sorts by the last key first: ratio descending, then p, then c.
    order = np.lexsort((c_v, p_v, -r_v.astype(np.float64)))
    cum = np.cumsum(cost[order])
    keep = order[cum <= budget(density, N)]        # costs > 0, so this is a prefix
    sel = np.zeros((Cq, Ck), dtype=bool)
    sel[p_v[keep], c_v[keep]] = True
    return sel


def compensated_attention(q, k, v, qa, ka, Ck: int, selected, scale: float, rows=None):
    """Output rows (float64 [R, d]) of compensated sparse attention, one (b, h)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    qa = np.asarray(qa, dtype=np.int64)
    ka = np.asarray(ka, dtype=np.int64)
    nk, kc = cluster_stats(k, ka, Ck)
    _, vc = cluster_stats(v, ka, Ck)
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    out = np.zeros((len(rows), v.shape[1]))
    for r, i in enumerate(rows):
        S = selected[qa[i]]                          # [Ck] selected key clusters
        exact = S[ka]                                # keys computed exactly
        virt = (~S) & (nk > 0)                       # clusters compensated
        l_exact = scale * (k[exact] @ q[i])
        l_virt = scale * (kc[virt] @ q[i]) + np.log(nk[virt])
        m = max(l_exact.max(initial=-np.inf), l_virt.max(initial=-np.inf))
        w_exact = np.exp(l_exact - m)
        w_virt = np.exp(l_virt - m)
        num = w_exact @ v[exact] + w_virt @ vc[virt]
        out[r] = num / (w_exact.sum() + w_virt.sum())
    return out


def centroid_attention(q, k, v, ka, Ck: int, scale: float, rows=None):
    """Closed form of density 0: o_i = sum_c n_c e^(s q_i.kc_c) vc_c / sum_c n_c e^(s q_i.kc_c)."""
    nk, kc = cluster_stats(k, ka, Ck)
    _, vc = cluster_stats(v, ka, Ck)
    q = np.asarray(q, dtype=np.float64)
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    nz = nk > 0
    out = np.zeros((len(rows), np.asarray(v).shape[1]))
    for r, i in enumerate(rows):
        a = scale * (kc[nz] @ q[i])
        w = nk[nz] * np.exp(a - a.max())
        out[r] = (w @ vc[nz]) / w.sum()
    return out
