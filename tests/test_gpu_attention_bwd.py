"""GPU block-sparse attention backward vs the float64 gradient oracle.

The forward runs on the GPU (its out and lse feed the backward, as in
training); the oracle recomputes everything from q, k, v and the upstream
gradient g in float64.

Tolerances, relative to the size of the reference because gradients are
O(1..10) where forward outputs are O(0.1):
* fp32: max |err| <= 1e-4 * max |want|;
* bf16: max |err| <= 3e-2 * max |want| and mean |err| <= 1e-2 * mean |want|.
  The bf16 output alone rounds each value by up to 2^-8 of itself (mean about
  2^-9); the bf16 P and dS operands of the tensor-core products and the bf16
  forward output behind delta add errors of the same relative order with
  random signs. The bar leaves a margin of about 3x and still fails on a
  dropped term, a wrong scale or a transposed operand by orders of magnitude.
"""
import numpy as np
import pytest
import torch

import synth
from conftest import cached_video_qkv
from oracle import attention as OA
from oracle import attention_bwd as OB
from oracle import masks as OM

pytestmark = pytest.mark.gpu


def assert_grad_close(got, want, dtype, what=""):
    got, want = np.asarray(got, dtype=np.float64), np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    assert np.isfinite(err).all(), "non-finite gradient " + what
    big, typ = np.abs(want).max(), np.abs(want).mean()
    if dtype == "f32":
        assert err.max() <= 1e-4 * big, (what, float(err.max()), float(big))
    else:
        assert err.max() <= 3e-2 * big, (what, float(err.max()), float(big))
        assert err.mean() <= 1e-2 * typ, (what, float(err.mean()), float(typ))


def _mask(va, kind, T, H, W, p, step=0):
    return va.mask_build(kind, T, H, W, block=p.block, w0=p.w0, local=p.local, period=p.period,
                         anchor0=p.anchor0, rot_stride=p.rot_stride, step=step)


def _gpu_grads(va, dev, q, k, v, g, m, scale, dtype):
    B, Hh, N, d = q.shape
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    qt, kt, vt, gt = (torch.from_numpy(x).to(dev, tdt) for x in (q, k, v, g))
    lse = torch.empty((B, Hh, N), dtype=torch.float32, device=dev)
    out, _ = va.sparse_attn_fwd(qt, kt, vt, m, scale=scale, lse=lse)
    dq, dk, dv = va.sparse_attn_bwd(qt, kt, vt, out, gt, lse, m, scale=scale)
    torch.cuda.synchronize()
    assert va.device_error() == va.OK
    return tuple(x.float().cpu().numpy() for x in (dq, dk, dv))


def _check(va, dev, q, k, v, g, kind, T, H, W, p, step, dtype, scale=None, rows=None, keys=None):
    d = q.shape[3]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    m = _mask(va, kind, T, H, W, p, step)
    got = _gpu_grads(va, dev, q, k, v, g, m, scale, dtype)
    m.free()
    bm = OM.block_mask(kind, T, H, W, p, step)
    want = OB.block_sparse_attention_grad(q, k, v, g, bm, p.block, scale, rows=rows, keys=keys)
    sel = (rows, keys, keys)
    for name, gg, ww, s in zip(("dq", "dk", "dv"), got, want, sel):
        assert_grad_close(gg if s is None else gg[:, :, s], ww, dtype, name)
    return got


def test_tiny_lvsa_fp32(va, dev):
    q, k, v = synth.iid_qkv(1, 2, 256, 64, seed=1235)
    g = synth.upstream_grad(1, 2, 256, 64, seed=1235, dtype="f32")
    _check(va, dev, q, k, v, g, OM.LVSA, 4, 8, 8, OM.MaskParams(block=64, local=1), 0, "f32",
           scale=0.125)


@pytest.mark.parametrize("d,block", [(64, 128), (128, 64), (128, 128)])
def test_fp32_other_shapes(va, dev, d, block):
    T, H, W = 5, 6, 11                                    # N = 330: ragged last block
    q, k, v = synth.iid_qkv(2, 2, T * H * W, d, seed=7)
    g = synth.upstream_grad(2, 2, T * H * W, d, seed=7, dtype="f32")
    _check(va, dev, q, k, v, g, OM.RADIAL, T, H, W, OM.MaskParams(block=block, w0=9), 0, "f32")


SMALL_BF16 = [
    (OM.RADIAL, 5, 6, 20, OM.MaskParams(block=128, w0=10), 0),          # N=600, tail 88
    (OM.RADIAL, 9, 8, 16, OM.MaskParams(block=128), 0),                 # N=1152, no tail
    (OM.LVSA, 12, 7, 9, OM.MaskParams(block=128, local=1, period=4, anchor0=2, rot_stride=3), 2),
    (OM.DENSE, 3, 7, 13, OM.MaskParams(block=128), 0),                 # N=273
    (OM.RADIAL, 1, 3, 5, OM.MaskParams(block=128), 0),                  # N=15 < block
]


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("case", SMALL_BF16)
def test_bf16_small_all_rows(va, dev, case, d):
    kind, T, H, W, p, step = case
    N = T * H * W
    q, k, v = synth.video_qkv(2, 3, T, H, W, d, seed=11)
    g = synth.upstream_grad(2, 3, N, d, seed=11)
    _check(va, dev, q, k, v, g, kind, T, H, W, p, step, "bf16")


# 64-token mask blocks on the tensor-core kernels: 128-token tiles over pairs
# of blocks with the dead 64 x 64 quarters zeroed; odd block counts and ragged
# tails, and an LVSA mask whose transposed lists differ from its rows
SMALL_BF16_B64 = [
    (OM.RADIAL, 5, 6, 20, OM.MaskParams(block=64, w0=10), 0),           # 10 blocks, tail 24
    (OM.LVSA, 12, 7, 9, OM.MaskParams(block=64, local=1, period=4, anchor0=2, rot_stride=3), 2),
    (OM.LVSA, 10, 8, 16, OM.MaskParams(block=64, local=0, period=3, anchor0=1, rot_stride=1), 1),
    (OM.DENSE, 3, 7, 13, OM.MaskParams(block=64), 0),                  # 5 blocks, tail 17
    (OM.RADIAL, 1, 3, 5, OM.MaskParams(block=64), 0),                   # N=15 < block
]


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("case", SMALL_BF16_B64)
def test_bf16_block64_small_all_rows(va, dev, case, d):
    kind, T, H, W, p, step = case
    N = T * H * W
    q, k, v = synth.video_qkv(1, 2, T, H, W, d, seed=17)
    g = synth.upstream_grad(1, 2, N, d, seed=17)
    _check(va, dev, q, k, v, g, kind, T, H, W, p, step, "bf16")


@pytest.mark.parametrize("d", [128, 64])
def test_bf16_other_scale_and_lvsa_asymmetry(va, dev, d):
    # LVSA's anchor frames make the block mask asymmetric, so the transposed
    # lists differ from the rows; a non-default scale checks where it enters.
    T, H, W = 10, 8, 16
    p = OM.MaskParams(block=128, local=0, period=3, anchor0=1, rot_stride=1)
    q, k, v = synth.video_qkv(1, 2, T, H, W, d, seed=13)
    g = synth.upstream_grad(1, 2, T * H * W, d, seed=13)
    bm = OM.block_mask(OM.LVSA, T, H, W, p, 1)
    assert not np.array_equal(bm, bm.T)
    _check(va, dev, q, k, v, g, OM.LVSA, T, H, W, p, 1, "bf16", scale=0.05)


def test_bf16_deterministic(va, dev):
    T, H, W = 6, 10, 13                                   # N = 780
    q, k, v = synth.video_qkv(1, 4, T, H, W, 128, seed=14)
    g = synth.upstream_grad(1, 4, T * H * W, 128, seed=14)
    m = va.mask_build(va.RADIAL, T, H, W)
    a = _gpu_grads(va, dev, q, k, v, g, m, 1 / np.sqrt(128), "bf16")
    b = _gpu_grads(va, dev, q, k, v, g, m, 1 / np.sqrt(128), "bf16")
    m.free()
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_wan_radial_full_size_sampled(va, dev):
    # The benchmarked workload: B=1, 12 heads, 21x30x52 = 32,760 tokens, d=128,
    # bf16, radial mask with block 128. dq on 256 sampled rows of every head;
    # dk and dv on sampled keys of the first block and the ragged last block of
    # head 0 (the oracle needs every query row that sees them); and over all
    # heads the softmax invariants sum_j dk_j = 0 and sum_j dv_j = sum_i g_i.
    T, H, W = 21, 30, 52
    N = T * H * W
    q, k, v = cached_video_qkv(1, 12, T, H, W, 128, seed=1235)
    g = synth.upstream_grad(1, 12, N, 128, seed=1235)
    p = OM.MaskParams(block=128)
    m = _mask(va, OM.RADIAL, T, H, W, p)
    dq, dk, dv = _gpu_grads(va, dev, q, k, v, g, m, 1 / np.sqrt(128), "bf16")
    m.free()
    bm = OM.block_mask(OM.RADIAL, T, H, W, p, 0)
    rows = OA.sample_rows(N, 128, 256, seed=6)
    want_dq, _, _ = OB.block_sparse_attention_grad(q, k, v, g, bm, 128, 1 / np.sqrt(128),
                                                   rows=rows, keys=np.array([], dtype=np.int64))
    assert_grad_close(dq[:, :, rows], want_dq, "bf16", "dq")
    last = (N - 1) // 128 * 128
    keys = np.array([0, 1, 77, 127, last, last + 5, N - 1])

    def mask_rows(r):
        return bm[(r // 128)[:, None], (np.arange(N) // 128)[None, :]]

    _, want_dk, want_dv = OB.attention_grad(q[0, 0], k[0, 0], v[0, 0], g[0, 0], mask_rows,
                                            1 / np.sqrt(128), rows=np.array([], dtype=np.int64),
                                            keys=keys)
    assert_grad_close(dk[0, 0, keys], want_dk, "bf16", "dk")
    assert_grad_close(dv[0, 0, keys], want_dv, "bf16", "dv")
    dk_sum = dk[0].astype(np.float64).sum(axis=1)                       # [heads, d]
    dv_sum = dv[0].astype(np.float64).sum(axis=1)
    g_sum = g[0].astype(np.float64).sum(axis=1)
    typical = np.abs(dk[0]).astype(np.float64).mean() * np.sqrt(N)     # random-walk size
    assert np.abs(dk_sum).max() <= 0.05 * typical
    assert np.abs(dv_sum - g_sum).max() <= 1e-2 * np.abs(g_sum).max() + 0.05 * np.abs(
        dv[0]).mean() * np.sqrt(N)


def test_backward_rejects_bad_arguments(va, dev):
    q = torch.zeros((1, 1, 240, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((1, 1, 240), dtype=torch.float32, device=dev)
    m = va.mask_build(va.RADIAL, 3, 4, 20)
    with pytest.raises(va.VAError) as e:                 # no lse
        va.sparse_attn_bwd(q, q, q, q, q, None, m)
    assert e.value.status == va.ERR_INVALID
    q96 = torch.zeros((1, 1, 240, 96), dtype=torch.bfloat16, device=dev)
    with pytest.raises(va.VAError) as e:                 # head_dim 96
        va.sparse_attn_bwd(q96, q96, q96, q96, q96, lse, m)
    assert e.value.status == va.ERR_UNSUPPORTED
    m2 = va.mask_build(va.RADIAL, 3, 4, 10)              # N mismatch
    with pytest.raises(va.VAError) as e:
        va.sparse_attn_bwd(q, q, q, q, q, lse, m2)
    assert e.value.status == va.ERR_INVALID
    assert va.device_error() == va.OK
