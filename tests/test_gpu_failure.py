"""Failure detection on the GPU without a fault: bounded device waits.

Every mbarrier wait in the library's kernels gives up after a clock64 limit,
records VA_ERR_TIMEOUT in a device error word and returns, instead of hanging
or trapping. va_selftest_wait_timeout runs that wait against a barrier no
thread arrives at; the status must come back through va_device_error and the
context must stay usable for the real kernels afterwards.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as OA
from oracle import masks as OM

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(va, dev):
    assert va.device_error() == va.OK
    va.selftest_wait_timeout(2_000_000)                  # about 1 ms at 2 GHz
    assert va.device_error() == va.ERR_TIMEOUT
    assert va.device_error() == va.OK                    # the word is cleared once read
    # the context still runs the attention kernel correctly
    T, H, W = 3, 4, 20
    q, k, v = synth.video_qkv(1, 2, T, H, W, 128, seed=77)
    m = va.mask_build(va.RADIAL, T, H, W, block=128, w0=6)
    qt, kt, vt = (torch.from_numpy(x).to(dev, torch.bfloat16) for x in (q, k, v))
    out, _ = va.sparse_attn_fwd(qt, kt, vt, m)
    assert va.device_error() == va.OK
    want, _ = OA.block_sparse_attention(q, k, v, OM.block_mask(OM.RADIAL, T, H, W,
                                                               OM.MaskParams(block=128, w0=6)),
                                        128, 1.0 / np.sqrt(128))
    assert np.abs(out.float().cpu().numpy() - want).max() <= 2e-2
    m.free()


def test_selftest_rejects_bad_limits(va):
    with pytest.raises(va.VAError):
        va.selftest_wait_timeout(10)
    with pytest.raises(va.VAError):
        va.selftest_wait_timeout(10 ** 11)
