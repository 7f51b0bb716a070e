"""Full-size long-sequence workloads on the GPU vs the float64 oracle (sampled rows).

* LVSA long horizon: B=1, 12 heads, 126 x 30 x 52 = 196,560 tokens (6x the
  Wan latent's 21 frames), d=128, bf16, +-2-frame local window plus a global
  anchor every 8th frame whose offset rotates with the denoising step
  (LVSA review, secrett2633 blog, sec. 3 and Fig. 2), steps 0..3.
* HunyuanVideo 720p shape: B=1, 24 heads, 33 x 45 x 80 = 118,800 tokens,
  d=128, bf16, radial mask, and the all-ones mask on the same kernel.

The oracle runs on 512 seeded query rows (always rows 0, N-1 and the first
row of the ragged last block) of every head; bars: max-abs <= 2e-2,
mean-abs <= 2e-3 on O, 2e-2 on LSE.
"""
import numpy as np
import pytest
import torch

from conftest import assert_bf16_close, cached_video_qkv
from oracle import attention as OA
from oracle import masks as OM

pytestmark = pytest.mark.gpu


def _check(va, dev, q, k, v, kind, T, H, W, p, step, rows):
    B, Hh, N, d = q.shape
    qt, kt, vt = (torch.from_numpy(x).to(dev, torch.bfloat16) for x in (q, k, v))
    m = va.mask_build(kind, T, H, W, block=p.block, w0=p.w0, local=p.local, period=p.period,
                      anchor0=p.anchor0, rot_stride=p.rot_stride, step=step)
    lse = torch.empty((B, Hh, N), dtype=torch.float32, device=dev)
    out, _ = va.sparse_attn_fwd(qt, kt, vt, m, lse=lse)
    assert va.device_error() == va.OK
    bm = OM.block_mask(kind, T, H, W, p, step)
    rp, col = m.csr()
    want_rp, want_col = OM.to_csr(bm)
    assert np.array_equal(rp, want_rp) and np.array_equal(col, want_col)
    m.free()
    got = out[:, :, torch.from_numpy(rows).to(dev)].float().cpu().numpy()
    got_lse = lse[:, :, torch.from_numpy(rows).to(dev)].cpu().numpy()
    del qt, kt, vt, out, lse
    torch.cuda.empty_cache()
    o_ref, lse_ref = OA.block_sparse_attention(q, k, v, bm, p.block, 1.0 / np.sqrt(d), rows=rows)
    assert_bf16_close(got, o_ref)
    assert np.abs(got_lse - lse_ref).max() <= 2e-2


@pytest.mark.parametrize("step", [0, 1, 2, 3])
def test_lvsa_long_horizon_rotating_anchors(va, dev, step):
    T, H, W = 126, 30, 52
    q, k, v = cached_video_qkv(1, 12, T, H, W, 128, seed=1237)
    rows = OA.sample_rows(T * H * W, 128, 512, seed=100 + step)
    p = OM.MaskParams(block=128, local=2, period=8, anchor0=0, rot_stride=1)
    _check(va, dev, q, k, v, OM.LVSA, T, H, W, p, step, rows)


@pytest.mark.parametrize("kind", [OM.RADIAL, OM.DENSE])
def test_hunyuan_720p(va, dev, kind):
    T, H, W = 33, 45, 80
    q, k, v = cached_video_qkv(1, 24, T, H, W, 128, seed=1239)
    rows = OA.sample_rows(T * H * W, 128, 512, seed=200 + kind)
    _check(va, dev, q, k, v, kind, T, H, W, OM.MaskParams(block=128), 0, rows)
