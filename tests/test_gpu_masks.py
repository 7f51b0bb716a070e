"""GPU mask builder vs the oracle: CSR lists must be bit-exact."""
import numpy as np
import pytest

from oracle import masks as OM

pytestmark = pytest.mark.gpu

R, L, D = OM.RADIAL, OM.LVSA, OM.DENSE

SMALL = [
    # kind, T, H, W, params, step
    (L, 4, 8, 8, OM.MaskParams(block=64, local=1), 0),                       # tiny LVSA check
    (R, 4, 1, 8, OM.MaskParams(block=4, w0=2), 0),
    (R, 5, 3, 7, OM.MaskParams(block=16), 0),
    (R, 9, 4, 4, OM.MaskParams(block=32, w0=3), 0),
    (R, 3, 1, 1, OM.MaskParams(block=2), 0),                                 # F = 1
    (R, 7, 5, 6, OM.MaskParams(block=64, w0=5), 0),
    (R, 40, 2, 3, OM.MaskParams(block=128, w0=6), 0),                        # block spans frames
    (L, 11, 2, 3, OM.MaskParams(block=8, local=2, period=3, anchor0=1, rot_stride=2), 1),
    (L, 10, 5, 5, OM.MaskParams(block=16, local=0, period=4, anchor0=-3, rot_stride=5), 7),
    (L, 6, 4, 4, OM.MaskParams(block=1, local=1, period=0, anchor0=5), 0),   # block 1
    (D, 3, 5, 7, OM.MaskParams(block=16), 0),
    (D, 1, 1, 1, OM.MaskParams(block=128), 0),                               # N = 1
    (R, 1, 3, 5, OM.MaskParams(block=128), 0),                               # N < block
]

FULL = [
    (R, 21, 30, 52, OM.MaskParams(block=128), 0),                            # Wan-shaped
    (L, 126, 30, 52, OM.MaskParams(block=128, local=2, period=8, rot_stride=1), 0),
    (L, 126, 30, 52, OM.MaskParams(block=128, local=2, period=8, rot_stride=1), 1),
    (L, 126, 30, 52, OM.MaskParams(block=128, local=2, period=8, rot_stride=1), 2),
    (L, 126, 30, 52, OM.MaskParams(block=128, local=2, period=8, rot_stride=1), 3),
    (R, 33, 45, 80, OM.MaskParams(block=128), 0),                            # HunyuanVideo 720p
    (D, 33, 45, 80, OM.MaskParams(block=128), 0),
]


def _build(va, kind, T, H, W, p, step):
    return va.mask_build(kind, T, H, W, block=p.block, w0=p.w0, local=p.local, period=p.period,
                         anchor0=p.anchor0, rot_stride=p.rot_stride, step=step)


@pytest.mark.parametrize("case", SMALL + FULL)
def test_mask_csr_bit_exact(va, case):
    kind, T, H, W, p, step = case
    m = _build(va, kind, T, H, W, p, step)
    rp, col = m.csr()
    bm = OM.block_mask(kind, T, H, W, p, step)
    want_rp, want_col = OM.to_csr(bm)
    assert m.nqb == bm.shape[0] and m.nnz == len(want_col)
    assert np.array_equal(rp, want_rp)
    assert np.array_equal(col, want_col)
    assert m.live_pairs == OM.live_pair_tokens(bm, p.block, T * H * W)
    m.free()
    assert va.device_error() == va.OK


def test_mask_rejects_bad_arguments(va):
    with pytest.raises(va.VAError) as e:
        va.mask_build(va.RADIAL, 0, 4, 4)
    assert e.value.status == va.ERR_INVALID
    with pytest.raises(va.VAError):
        va.mask_build(va.RADIAL, 4, 4, 4, block=0)
    with pytest.raises(va.VAError):
        va.mask_build(va.LVSA, 4, 4, 4, period=-1)
    with pytest.raises(va.VAError):
        va.mask_build(7, 4, 4, 4)
    with pytest.raises(va.VAError):
        va.mask_build(va.RADIAL, 1 << 12, 1 << 10, 1 << 9)       # N >= 2^30


def test_mask_allocation_failure_is_reported(va, monkeypatch):
    monkeypatch.setenv("VA_FAULT_INJECT", "alloc")
    with pytest.raises(va.VAError) as e:
        va.mask_build(va.RADIAL, 4, 4, 4)
    assert e.value.status == va.ERR_OOM
    monkeypatch.delenv("VA_FAULT_INJECT")
    m = va.mask_build(va.RADIAL, 4, 4, 4, block=16)
    assert m.nnz > 0


def test_mask_limits_on_blocks_and_live_pairs(va):
    # At most VA_MASK_MAX_BLOCKS = 65,536 blocks per side. The dense mask of
    # 65,536 one-token blocks has 2^32 live block pairs, more than int32 row
    # offsets can index: the build stops after counting, before any list is
    # filled or sized, and reports the grid as unsupported.
    with pytest.raises(va.VAError) as e:
        va.mask_build(va.DENSE, 1, 1, 65537, block=1)
    assert e.value.status == va.ERR_UNSUPPORTED
    with pytest.raises(va.VAError) as e:
        va.mask_build(va.DENSE, 1, 1, 65536, block=1)
    assert e.value.status == va.ERR_UNSUPPORTED
    assert va.device_error() == va.OK
    m = va.mask_build(va.DENSE, 1, 1, 4096, block=1)              # works again afterwards
    assert m.nnz == 4096 * 4096
    m.free()
    assert va.device_error() == va.OK


@pytest.mark.parametrize("case", SMALL[:6] + FULL)
def test_checked_mode_validates_built_masks(va, case, monkeypatch):
    # With VA_CHECKED set, va_mask_build copies its rows and transposed lists
    # back and validates them (CSR rules, diagonal, exact transpose).
    monkeypatch.setenv("VA_CHECKED", "1")
    kind, T, H, W, p, step = case
    m = _build(va, kind, T, H, W, p, step)
    rp, col = m.csr()
    assert va.csr_validate(rp, col) == va.OK
    m.free()
    assert va.device_error() == va.OK


def _cache_get(cache, kind, T, H, W, p, step):
    return cache.get(kind, T, H, W, block=p.block, w0=p.w0, local=p.local, period=p.period,
                     anchor0=p.anchor0, rot_stride=p.rot_stride, step=step)


def test_mask_cache_reuse_is_bit_exact(va):
    """Cached masks across denoising steps: one entry per LVSA rotation phase,
    one radial mask for every step, each CSR equal to the oracle's at the
    requested step."""
    import torch
    cache = va.MaskCache(capacity=8)
    T, H, W = 11, 4, 5
    p = OM.MaskParams(block=16, local=1, period=3, anchor0=1, rot_stride=1)
    handles = {}
    for step in range(8):
        m = _cache_get(cache, L, T, H, W, p, step)
        rp, col = m.csr()
        want_rp, want_col = OM.to_csr(OM.block_mask(L, T, H, W, p, step))
        assert np.array_equal(rp, want_rp) and np.array_equal(col, want_col), step
        handles[step] = m.handle.value
    assert handles[0] == handles[3] == handles[6]
    assert len({handles[0], handles[1], handles[2]}) == 3
    assert cache.stats() == (5, 3, 3)
    pr = OM.MaskParams(block=64)
    r0 = _cache_get(cache, R, 4, 8, 8, pr, 0)
    r1 = _cache_get(cache, R, 4, 8, 8, pr, 9)
    assert r0.handle.value == r1.handle.value
    assert cache.stats() == (6, 4, 4)
    # a cached mask drives attention exactly as a freshly built one
    g = torch.Generator(device="cuda").manual_seed(5)
    q, k, v = (torch.randn(1, 2, 256, 128, device="cuda", generator=g).to(torch.bfloat16)
               for _ in range(3))
    fresh = _build(va, R, 4, 8, 8, pr, 3)
    oa, _ = va.sparse_attn_fwd(q, k, v, r1)
    ob, _ = va.sparse_attn_fwd(q, k, v, fresh)
    torch.cuda.synchronize()
    assert torch.equal(oa, ob)
    fresh.free()
    r1.free()  # a cached mask's free() leaves the mask to the cache
    oc, _ = va.sparse_attn_fwd(q, k, v, r0)
    torch.cuda.synchronize()
    assert torch.equal(oc, oa)
    cache.clear()
    with pytest.raises(va.VAError):
        r0.handle
    assert cache.stats()[2] == 0
    again = _cache_get(cache, L, T, H, W, p, 4)
    assert np.array_equal(again.csr()[1], OM.to_csr(OM.block_mask(L, T, H, W, p, 4))[1])
    cache.close()
    with pytest.raises(va.VAError):
        again.handle
    assert va.device_error() == va.OK


def test_mask_cache_full_builds_nothing(va):
    cache = va.MaskCache(capacity=2)
    for w0 in (1, 2):
        _cache_get(cache, R, 4, 2, 2, OM.MaskParams(block=4, w0=w0), 0)
    with pytest.raises(va.VAError) as e:
        _cache_get(cache, R, 4, 2, 2, OM.MaskParams(block=4, w0=3), 0)
    assert e.value.status == va.ERR_UNSUPPORTED
    _cache_get(cache, R, 4, 2, 2, OM.MaskParams(block=4, w0=1), 5)  # a hit still works
    assert cache.stats() == (1, 2, 2)
    cache.close()
