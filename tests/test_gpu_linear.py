"""GPU linear attention and LinVideo's mixed attention vs the float64 oracle.

Bars: the bf16 attention bars (max-abs 2e-2, mean-abs 2e-3). Readings of
LinVideo (gist.science 2510.08318), technical summary secs. 1 and 2 A: feature
map elu(x) + 1, non-causal, mix = r * attention + (1 - r) * linear.
"""
import numpy as np
import pytest
import torch

import synth
from conftest import assert_bf16_close, cached_video_qkv
from oracle import attention as OA
from oracle import linear as OL
from oracle import masks as OM

pytestmark = pytest.mark.gpu


def _dev(x, dev):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev, torch.bfloat16)


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("B,Hh,T,H,W", [(2, 2, 5, 6, 11),     # N = 330: ragged tail tile
                                        (1, 3, 1, 7, 13),     # N = 91 < one tile
                                        (1, 1, 3, 43, 1),     # N = 129: one token past a tile
                                        (2, 80, 2, 8, 8)])    # 160 slices: one split each
def test_linear_small(va, dev, B, Hh, T, H, W, d):
    N = T * H * W
    q, k, v = synth.video_qkv(B, Hh, T, H, W, d, seed=41, dtype="bf16")
    out = va.linear_attn_fwd(_dev(q, dev), _dev(k, dev), _dev(v, dev))
    torch.cuda.synchronize()
    assert va.device_error() == va.OK
    want = OL.linear_attention(q, k, v)
    assert_bf16_close(out.float().cpu().numpy(), want)


def test_linear_identical_keys_give_mean_value(va, dev):
    T, H, W = 4, 8, 9
    N = T * H * W
    q, k, v = synth.video_qkv(1, 2, T, H, W, 128, seed=43, dtype="bf16")
    k = np.ascontiguousarray(np.broadcast_to(k[:, :, :1], k.shape))
    out = va.linear_attn_fwd(_dev(q, dev), _dev(k, dev), _dev(v, dev))
    torch.cuda.synchronize()
    want = np.broadcast_to(v.astype(np.float64).mean(axis=2, keepdims=True), v.shape)
    assert_bf16_close(out.float().cpu().numpy(), want)


@pytest.mark.parametrize("d", [128, 64])
def test_linear_extreme_feature_inputs(va, dev, d):
    # phi(-inf) = 0 and phi of large negative inputs underflows to 0; large
    # positive inputs give x + 1. Some dims of Q and K take such values (no
    # row is all -inf, so every denominator stays positive).
    T, H, W = 3, 7, 13
    q, k, v = synth.video_qkv(1, 2, T, H, W, d, seed=47, dtype="bf16")
    q, k = q.copy(), k.copy()
    k[:, :, ::3, 5] = -np.inf
    k[:, :, 1::4, 7] = -300.0
    k[:, :, 2::5, 9] = -40.0
    k[:, :, ::7, 11] = 30.0
    q[:, :, ::2, 3] = -np.inf
    q[:, :, 1::3, 4] = -90.0
    q[:, :, ::5, 6] = 20.0
    out = va.linear_attn_fwd(_dev(q, dev), _dev(k, dev), _dev(v, dev))
    torch.cuda.synchronize()
    assert va.device_error() == va.OK
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert_bf16_close(got, OL.linear_attention(q, k, v))


@pytest.mark.parametrize("d", [128, 64])
def test_linear_full_size(va, dev, d):
    # Wan-shaped inputs: B=1, 12 heads, 21x30x52 = 32,760 tokens, bf16, with
    # head_dim 128 and 64; the oracle on 512 sampled rows of every head
    T, H, W = 21, 30, 52
    N = T * H * W
    q, k, v = cached_video_qkv(1, 12, T, H, W, d, seed=1235)
    out = va.linear_attn_fwd(_dev(q, dev), _dev(k, dev), _dev(v, dev))
    torch.cuda.synchronize()
    assert va.device_error() == va.OK
    rows = OA.sample_rows(N, 128, 512, seed=21)
    got = out[:, :, torch.from_numpy(rows).to(dev)].float().cpu().numpy()
    assert_bf16_close(got, OL.linear_attention(q, k, v, rows=rows))


@pytest.mark.parametrize("r,d", [(0.0, 128), (0.3, 128), (1.0, 128), (0.0, 64), (0.3, 64)])
def test_mixed(va, dev, r, d):
    T, H, W = 5, 6, 11
    N = T * H * W
    q, k, v = synth.video_qkv(1, 3, T, H, W, d, seed=47, dtype="bf16")
    p = OM.MaskParams(block=128, w0=9)
    m = va.mask_build(OM.RADIAL, T, H, W, block=128, w0=9)
    qt, kt, vt = _dev(q, dev), _dev(k, dev), _dev(v, dev)
    out = va.mixed_attn_fwd(qt, kt, vt, m, r)
    torch.cuda.synchronize()
    assert va.device_error() == va.OK
    bm = OM.block_mask(OM.RADIAL, T, H, W, p, 0)
    want = OL.mixed_attention(q, k, v, bm, 128, 1.0 / np.sqrt(d), r)
    assert_bf16_close(out.float().cpu().numpy(), want)
    if r == 1.0:   # the attention alone, bit for bit
        att, _ = va.sparse_attn_fwd(qt, kt, vt, m)
        assert torch.equal(out, att)
    if r == 0.0:   # the linear attention alone, bit for bit
        assert torch.equal(out, va.linear_attn_fwd(qt, kt, vt))
    m.free()


def test_mixed_rejects_bad_arguments(va, dev):
    q = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16, device=dev)
    m = va.mask_build(OM.RADIAL, 1, 8, 8, block=128)
    for r in (-0.1, 1.5, float("nan")):
        with pytest.raises(va.VAError):
            va.mixed_attn_fwd(q, q, q, m, r)
    with pytest.raises(va.VAError):
        va.linear_attn_fwd(q.float(), q.float(), q.float())
    q32 = torch.zeros((1, 1, 64, 32), dtype=torch.bfloat16, device=dev)
    with pytest.raises(va.VAError) as e:       # head_dim 64 and 128 only
        va.linear_attn_fwd(q32, q32, q32)
    assert e.value.status == va.ERR_UNSUPPORTED
    m.free()
