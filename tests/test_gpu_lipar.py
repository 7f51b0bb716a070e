"""GPU LIPAR pruning / restoration vs the oracle (readings of the LIPAR summary,
sec. 2 B). Pruning decisions are integers taken on exact float32 differences:
keep, order, count and src must match bit for bit. Gather and restore are
copies: exact. Prune -> gather -> attention -> restore is compared with the
oracle's composition at the bf16 attention bars.

Latent recipe (seeded): B clips of T x H x W tokens with C = 16 channels (the
Wan VAE latent width); a static N(0, 1) background with per-frame jitter of
amplitude tau / 4 (below the threshold), plus a square of side 3 that moves by
one cell per frame and gets fresh N(0, 1) values where it is.
"""
import numpy as np
import pytest
import torch

from conftest import assert_bf16_close
from oracle import attention as OA
from oracle import lipar as OLP
from oracle import masks as OM

pytestmark = pytest.mark.gpu

TAU = 0.5


def _latent(B, T, H, W, C, seed):
    rng = np.random.default_rng(seed)
    x = np.repeat(rng.normal(size=(B, 1, H, W, C)), T, axis=1)
    x += rng.uniform(-TAU / 4, TAU / 4, size=x.shape)
    for b in range(B):
        for t in range(T):
            h0, w0 = (2 + t) % (H - 2), (1 + 2 * t + b) % (W - 2)
            x[b, t, h0:h0 + 3, w0:w0 + 3] = rng.normal(size=(3, 3, C))
    # bf16-representable values, so both sides see the same numbers
    x = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy()
    return x.reshape(B, T * H * W, C)


@pytest.mark.parametrize("B,T,H,W,dtype", [(2, 9, 12, 20, "bf16"), (1, 5, 7, 9, "f32"),
                                           (1, 21, 30, 52, "bf16")])   # Wan latent grid
def test_prune_matches_oracle(va, dev, B, T, H, W, dtype):
    C = 16
    x = _latent(B, T, H, W, C, seed=61 + T)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    keep, order, src, count = va.lipar_prune(torch.from_numpy(x).to(dev, tdt), T, H, W, TAU)
    torch.cuda.synchronize()
    assert va.device_error() == va.OK
    keep, order, src, count = (t.cpu().numpy() for t in (keep, order, src, count))
    for b in range(B):
        k_w, o_w, s_w, n_w = OLP.prune(x[b], T, H, W, TAU)
        assert count[b] == n_w
        assert np.array_equal(keep[b].astype(bool), k_w)
        assert np.array_equal(order[b, :n_w], o_w)
        assert np.array_equal(src[b], s_w)
        assert H * W <= n_w < T * H * W      # something was pruned, frame 0 kept


def test_gather_restore_are_exact_copies(va, dev):
    B, T, H, W, Hh, d = 2, 6, 8, 10, 3, 128
    N = T * H * W
    x = _latent(B, T, H, W, 16, seed=71)
    _, order, src, count = va.lipar_prune(torch.from_numpy(x).to(dev, torch.bfloat16), T, H, W,
                                          TAU)
    y = torch.randn((B, Hh, N, d), device=dev).to(torch.bfloat16)
    yc = va.lipar_gather(y, order, count)
    full = va.lipar_restore(yc, src)
    torch.cuda.synchronize()
    o, s, n = order.cpu().numpy(), src.cpu().numpy(), count.cpu().numpy()
    yn, ycn, fn = y.float().cpu().numpy(), yc.float().cpu().numpy(), full.float().cpu().numpy()
    for b in range(B):
        assert np.array_equal(ycn[b, :, :n[b]], yn[b][:, o[b, :n[b]]])
        assert np.array_equal(fn[b], ycn[b][:, s[b]])


def test_pruned_attention_matches_oracle_composition(va, dev):
    # prune the latent, run dense attention on the kept tokens, restore
    T, H, W, Hh, d = 7, 10, 14, 2, 128
    N = T * H * W
    x = _latent(1, T, H, W, 16, seed=81)
    _, order, src, count = va.lipar_prune(torch.from_numpy(x).to(dev, torch.bfloat16), T, H, W,
                                          TAU)
    rng = np.random.default_rng(82)
    qkv = [torch.from_numpy(rng.normal(size=(1, Hh, N, d)).astype(np.float32)).to(torch.bfloat16)
           for _ in range(3)]
    qc, kc, vc = (va.lipar_gather(t.to(dev), order, count) for t in qkv)
    n = int(count.item())
    m = va.mask_build(OM.DENSE, 1, 1, n, block=128)
    oc, _ = va.sparse_attn_fwd(qc[:, :, :n].contiguous(), kc[:, :, :n].contiguous(),
                               vc[:, :, :n].contiguous(), m)
    padded = torch.zeros((1, Hh, N, d), dtype=torch.bfloat16, device=dev)
    padded[:, :, :n] = oc
    full = va.lipar_restore(padded, src)
    torch.cuda.synchronize()
    assert va.device_error() == va.OK
    m.free()
    _, o_w, s_w, n_w = OLP.prune(x[0], T, H, W, TAU)
    q, k, v = (t.float().numpy()[0] for t in qkv)
    want = np.empty((Hh, N, d))
    for h in range(Hh):
        att, _ = OA.attention_rows(q[h][o_w], k[h][o_w], v[h][o_w],
                                   lambda r: np.ones((len(r), n_w), dtype=bool), 1 / np.sqrt(d))
        want[h] = OLP.restore(att, s_w)
    assert_bf16_close(full.float().cpu().numpy()[0], want)


def test_prune_rejects_bad_arguments(va, dev):
    x = torch.zeros((1, 2 * 3 * 4, 8), dtype=torch.bfloat16, device=dev)
    with pytest.raises(va.VAError):
        va.lipar_prune(x, 2, 3, 5, TAU)           # N != T*H*W
    with pytest.raises(va.VAError):
        va.lipar_prune(x, 2, 3, 4, float("nan"))
