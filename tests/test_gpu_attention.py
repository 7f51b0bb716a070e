"""GPU block-sparse attention vs the float64 oracle.

bf16 inputs: max-abs <= 2e-2 and mean-abs <= 2e-3; fp32 inputs: max-abs <= 1e-4.
Small cases are compared on every output; full-size workloads on 512 seeded
sampled query rows (always including rows 0, N-1 and the first row of the
ragged last block) of every (batch, head).
"""
import numpy as np
import pytest
import torch

import synth
from conftest import assert_bf16_close, cached_video_qkv
from oracle import attention as OA
from oracle import masks as OM

pytestmark = pytest.mark.gpu


def _mask(va, kind, T, H, W, p, step=0):
    return va.mask_build(kind, T, H, W, block=p.block, w0=p.w0, local=p.local, period=p.period,
                         anchor0=p.anchor0, rot_stride=p.rot_stride, step=step)


def _run(va, dev, q, k, v, kind, T, H, W, p, step, dtype, rows=None, scale=None):
    B, Hh, N, d = q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    qt, kt, vt = (torch.from_numpy(x).to(dev, tdt) for x in (q, k, v))
    m = _mask(va, kind, T, H, W, p, step)
    lse = torch.empty((B, Hh, N), dtype=torch.float32, device=dev)
    out, _ = va.sparse_attn_fwd(qt, kt, vt, m, scale=scale, lse=lse)
    assert va.device_error() == va.OK
    bm = OM.block_mask(kind, T, H, W, p, step)
    o_ref, lse_ref = OA.block_sparse_attention(q, k, v, bm, p.block, scale, rows=rows)
    got = out.float().cpu().numpy()
    got_lse = lse.cpu().numpy()
    if rows is not None:
        got, got_lse = got[:, :, rows], got_lse[:, :, rows]
    m.free()
    return got, o_ref, got_lse, lse_ref


def test_tiny_lvsa_fp32(va, dev):
    # B=1, 2 heads, 4 frames of 8x8, d=64, i.i.d. N(0,1) fp32, block 64,
    # +-1 frame window + anchor frame 0, scale 1/8.
    q, k, v = synth.iid_qkv(1, 2, 256, 64, seed=1235)
    got, want, gl, wl = _run(va, dev, q, k, v, OM.LVSA, 4, 8, 8, OM.MaskParams(block=64, local=1),
                             0, "f32", scale=0.125)
    assert np.abs(got - want).max() <= 1e-4
    assert np.abs(gl - wl).max() <= 1e-4


@pytest.mark.parametrize("d,block", [(64, 128), (128, 64), (128, 128)])
def test_fp32_other_shapes(va, dev, d, block):
    T, H, W = 5, 6, 11                                    # N = 330: ragged last block
    q, k, v = synth.iid_qkv(2, 2, T * H * W, d, seed=7)
    got, want, gl, wl = _run(va, dev, q, k, v, OM.RADIAL, T, H, W, OM.MaskParams(block=block, w0=9),
                             0, "f32")
    assert np.abs(got - want).max() <= 1e-4
    assert np.abs(gl - wl).max() <= 1e-4


SMALL_BF16 = [
    (OM.RADIAL, 5, 6, 20, OM.MaskParams(block=128, w0=10), 0),          # N=600, tail 88
    (OM.RADIAL, 9, 8, 16, OM.MaskParams(block=128), 0),                 # N=1152, no tail
    (OM.LVSA, 12, 7, 9, OM.MaskParams(block=128, local=1, period=4, anchor0=2, rot_stride=3), 2),
    (OM.DENSE, 3, 7, 13, OM.MaskParams(block=128), 0),                 # N=273
    (OM.RADIAL, 1, 3, 5, OM.MaskParams(block=128), 0),                  # N=15 < block
    (OM.DENSE, 1, 1, 1, OM.MaskParams(block=128), 0),                   # N=1
]


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("case", SMALL_BF16)
def test_bf16_small_all_rows(va, dev, case, d):
    kind, T, H, W, p, step = case
    q, k, v = synth.video_qkv(2, 3, T, H, W, d, seed=11)
    got, want, gl, wl = _run(va, dev, q, k, v, kind, T, H, W, p, step, "bf16")
    assert_bf16_close(got, want)
    assert np.abs(gl - wl).max() <= 2e-2


# 64-token mask blocks on the tensor-core kernel: 128-row tiles over pairs of
# query blocks, entries over pairs of key blocks, dead 64 x 64 quarters masked
SMALL_BF16_B64 = [
    (OM.RADIAL, 5, 6, 20, OM.MaskParams(block=64, w0=10), 0),           # 10 blocks, tail 24
    (OM.RADIAL, 9, 8, 16, OM.MaskParams(block=64), 0),                  # 18 blocks, no tail
    (OM.LVSA, 12, 7, 9, OM.MaskParams(block=64, local=1, period=4, anchor0=2, rot_stride=3), 2),
    (OM.LVSA, 16, 4, 8, OM.MaskParams(block=64, local=0, period=5, anchor0=1, rot_stride=2), 1),
    (OM.DENSE, 3, 7, 13, OM.MaskParams(block=64), 0),                  # 5 blocks, tail 17
    (OM.RADIAL, 3, 4, 20, OM.MaskParams(block=64, w0=7), 0),            # 4 blocks, tail 48
    (OM.RADIAL, 1, 3, 5, OM.MaskParams(block=64), 0),                   # N=15 < block
]


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("case", SMALL_BF16_B64)
def test_bf16_block64_small_all_rows(va, dev, case, d):
    kind, T, H, W, p, step = case
    q, k, v = synth.video_qkv(2, 3, T, H, W, d, seed=13)
    got, want, gl, wl = _run(va, dev, q, k, v, kind, T, H, W, p, step, "bf16")
    assert_bf16_close(got, want)
    assert np.abs(gl - wl).max() <= 2e-2


def test_bf16_block64_wan_sampled_rows(va, dev):
    # The Wan grid (32,760 tokens, 12 heads, d=128) under the radial mask with
    # 64-token blocks (512 blocks; W0 = H*W)
    T, H, W = 21, 30, 52
    q, k, v = cached_video_qkv(1, 12, T, H, W, 128, seed=1235)
    rows = OA.sample_rows(T * H * W, 64, 512, seed=6)
    got, want, gl, wl = _run(va, dev, q, k, v, OM.RADIAL, T, H, W, OM.MaskParams(block=64),
                             0, "bf16", rows=rows)
    assert_bf16_close(got, want)
    assert np.abs(gl - wl).max() <= 2e-2


def test_bf16_single_live_key_block_extremes(va, dev):
    # Large-magnitude logits (scale 1): the online softmax must stay finite.
    T, H, W = 4, 8, 16
    q, k, v = synth.video_qkv(1, 2, T, H, W, 128, seed=12)
    got, want, gl, wl = _run(va, dev, q * 4, k * 4, v, OM.RADIAL, T, H, W,
                             OM.MaskParams(block=128, w0=3), 0, "bf16", scale=1.0)
    assert_bf16_close(got, want)


def _bf16_exact(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).bfloat16().float().numpy()


@pytest.mark.parametrize("d,block", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_bf16_negative_scale(va, dev, d, block):
    # sl2 < 0: the max pass takes the smallest raw logit
    T, H, W = 3, 5, 20
    q, k, v = synth.video_qkv(1, 2, T, H, W, d, seed=14)
    got, want, gl, wl = _run(va, dev, q, k, v, OM.RADIAL, T, H, W, OM.MaskParams(block=block),
                             0, "bf16", scale=-1.0 / np.sqrt(d))
    assert_bf16_close(got, want)
    assert np.abs(gl - wl).max() <= 2e-2


@pytest.mark.parametrize("d,block", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_bf16_running_max_rises_every_block(va, dev, d, block):
    # Every query points along u and key j's component along u grows with j,
    # so each key block raises the row max by about 25 (log2 units): past the
    # rescale threshold, every block takes the max pass and rescales O.
    T, H, W = 4, 16, 16
    N = T * H * W
    rng = np.random.default_rng(15)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    q = 8.0 * u[None, :] + 0.05 * rng.standard_normal((N, d))
    k = (200.0 * np.arange(N) / N)[:, None] * u[None, :] + 0.05 * rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    q, k, v = (_bf16_exact(x.reshape(1, 1, N, d)) for x in (q, k, v))
    got, want, gl, wl = _run(va, dev, q, k, v, OM.DENSE, T, H, W, OM.MaskParams(block=block),
                             0, "bf16")
    assert np.isfinite(got).all()
    assert_bf16_close(got, want)
    assert np.abs(gl - wl).max() <= 2e-2


@pytest.mark.parametrize("d", [128, 64])
def test_wan_radial_full_size_sampled_rows(va, dev, d):
    # The benchmarked workload: B=1, 12 heads, 21x30x52 = 32,760 tokens, d=128,
    # bf16, radial mask with block 128 (W0 = H*W); and the same grid with d=64.
    T, H, W = 21, 30, 52
    q, k, v = cached_video_qkv(1, 12, T, H, W, d, seed=1235)
    rows = OA.sample_rows(T * H * W, 128, 512, seed=5)
    got, want, gl, wl = _run(va, dev, q, k, v, OM.RADIAL, T, H, W, OM.MaskParams(block=128),
                             0, "bf16", rows=rows)
    assert_bf16_close(got, want)
    assert np.abs(gl - wl).max() <= 2e-2


def test_attention_rejects_bad_arguments(va, dev):
    q = torch.zeros((1, 1, 240, 128), dtype=torch.bfloat16, device=dev)
    m = va.mask_build(va.RADIAL, 3, 4, 20)
    with pytest.raises(va.VAError) as e:                 # N mismatch
        va.sparse_attn_fwd(q[:, :, :200].contiguous(), q[:, :, :200].contiguous(),
                           q[:, :, :200].contiguous(), m)
    assert e.value.status == va.ERR_INVALID
    q96 = torch.zeros((1, 1, 240, 96), dtype=torch.bfloat16, device=dev)
    with pytest.raises(va.VAError) as e:                 # head_dim 96
        va.sparse_attn_fwd(q96, q96, q96, m)
    assert e.value.status == va.ERR_UNSUPPORTED
    assert va.device_error() == va.OK


@pytest.mark.parametrize("pinned,with_lse,dtype,d", [(True, True, "bf16", 128),
                                                     (False, False, "bf16", 128),
                                                     (True, True, "f32", 128),
                                                     (True, True, "bf16", 64)])
def test_host_buffers_match_device_call(va, dev, pinned, with_lse, dtype, d):
    # va_sparse_attn_fwd_host (host q/k/v/out, pipelined chunks) must give the
    # device call's result bit for bit: every (batch, head) runs the same kernel.
    T, H, W = 5, 6, 11                                    # N = 330: ragged last block
    B, Hh = 3, 5                                          # 15 slices: chunks of one slice
    q, k, v = synth.iid_qkv(B, Hh, T * H * W, d, seed=17)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    qh, kh, vh = (torch.from_numpy(x).to(tdt) for x in (q, k, v))
    if pinned:
        qh, kh, vh = qh.pin_memory(), kh.pin_memory(), vh.pin_memory()
    m = _mask(va, OM.RADIAL, T, H, W, OM.MaskParams(block=128, w0=9))
    lse_d = torch.empty((B, Hh, T * H * W), dtype=torch.float32, device=dev) if with_lse else None
    out_d, _ = va.sparse_attn_fwd(qh.to(dev), kh.to(dev), vh.to(dev), m, lse=lse_d)
    lse_h = torch.empty((B, Hh, T * H * W), dtype=torch.float32) if with_lse else None
    if with_lse and pinned:
        lse_h = lse_h.pin_memory()
    out_h, _ = va.sparse_attn_fwd_host(qh, kh, vh, m, lse=lse_h)
    torch.cuda.synchronize()
    assert va.device_error() == va.OK
    assert torch.equal(out_h, out_d.cpu())
    if with_lse:
        assert torch.equal(lse_h, lse_d.cpu())
    m.free()


def test_host_buffers_full_size(va, dev):
    # Wan-shaped radial workload through the host entry, bit-exact against the
    # device call (12 slices, one per chunk).
    T, H, W = 21, 30, 52
    q, k, v = cached_video_qkv(1, 12, T, H, W, 128, seed=1235)
    qh, kh, vh = (torch.from_numpy(x).to(torch.bfloat16).pin_memory() for x in (q, k, v))
    m = _mask(va, OM.RADIAL, T, H, W, OM.MaskParams(block=128))
    out_d, _ = va.sparse_attn_fwd(qh.to(dev), kh.to(dev), vh.to(dev), m)
    out_h, _ = va.sparse_attn_fwd_host(qh, kh, vh, m)
    torch.cuda.synchronize()
    assert va.device_error() == va.OK
    assert torch.equal(out_h, out_d.cpu())
    m.free()
