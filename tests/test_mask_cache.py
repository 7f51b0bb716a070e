"""The mask cache's key, pinned on the CPU against the oracle's masks.

A cache entry serves every request whose key matches, so the key must never
join two requests whose block masks differ (the cache would hand out a wrong
mask); the cases below also hold pairs it must join (the radial mask at any
step, LVSA steps a rotation period apart). No GPU: va_mask_same is host-only.
"""
import ctypes
import os

import numpy as np
import pytest

from oracle import masks as OM

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, ERR_INVALID, ERR_UNSUPPORTED = 0, -1, -2

R, L, D = OM.RADIAL, OM.LVSA, OM.DENSE


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__._build_module().build()
    lib = ctypes.CDLL(os.path.join(ROOT, "linear_attention_video_fwd_b300", "libva.so"))
    return lib


class _P(ctypes.Structure):
    _fields_ = [("block", ctypes.c_int32), ("w0", ctypes.c_int32), ("local", ctypes.c_int32),
                ("period", ctypes.c_int32), ("anchor0", ctypes.c_int32),
                ("rot_stride", ctypes.c_int32)]


def _same(lib, kind, T, H, W, p, sa, sb):
    cp = _P(p.block, p.w0, p.local, p.period, p.anchor0, p.rot_stride)
    out = ctypes.c_int(-1)
    st = lib.va_mask_same(kind, T, H, W, ctypes.byref(cp), sa, sb, ctypes.byref(out))
    return st, out.value


CASES = [
    (R, 9, 2, 3, OM.MaskParams(block=4, w0=2)),
    (R, 6, 3, 3, OM.MaskParams(block=8)),
    (D, 5, 2, 2, OM.MaskParams(block=4, period=3, anchor0=1)),
    (L, 9, 2, 3, OM.MaskParams(block=4, local=1, period=3, anchor0=1, rot_stride=1)),
    (L, 10, 2, 2, OM.MaskParams(block=2, local=0, period=4, anchor0=-3, rot_stride=2)),
    (L, 12, 1, 3, OM.MaskParams(block=3, local=1, period=5, anchor0=7, rot_stride=-3)),
    (L, 8, 2, 2, OM.MaskParams(block=4, local=0, period=0, anchor0=5, rot_stride=1)),
    (L, 7, 2, 2, OM.MaskParams(block=8, local=2, period=2, anchor0=0, rot_stride=1)),
]
STEPS = range(0, 9)


@pytest.mark.parametrize("case", CASES)
def test_shared_entries_have_identical_masks(lib, case):
    kind, T, H, W, p = case
    masks = {s: OM.block_mask_literal(kind, T, H, W, p, s) for s in STEPS}
    for sa in STEPS:
        for sb in STEPS:
            st, same = _same(lib, kind, T, H, W, p, sa, sb)
            assert st == OK
            if same:
                assert np.array_equal(masks[sa], masks[sb]), (case, sa, sb)
            if sa == sb:
                assert same == 1


def test_cases_exercise_both_outcomes(lib):
    joined = split_differ = 0
    for kind, T, H, W, p in CASES:
        for sa in STEPS:
            for sb in STEPS:
                if sa == sb:
                    continue
                _, same = _same(lib, kind, T, H, W, p, sa, sb)
                if same:
                    joined += 1
                elif not np.array_equal(OM.block_mask_literal(kind, T, H, W, p, sa),
                                        OM.block_mask_literal(kind, T, H, W, p, sb)):
                    split_differ += 1
    assert joined > 0 and split_differ > 0


def test_reuse_rules(lib):
    # radial and dense masks: one entry for every step; LVSA: period phases
    _, same = _same(lib, R, 9, 2, 3, OM.MaskParams(block=4), 0, 41)
    assert same == 1
    p = OM.MaskParams(block=4, local=1, period=3, anchor0=1, rot_stride=1)
    assert _same(lib, L, 9, 2, 3, p, 2, 5)[1] == 1
    assert _same(lib, L, 9, 2, 3, p, 2, 4)[1] == 0
    # phase of a negative product wraps like the mask rule
    p = OM.MaskParams(block=4, local=0, period=4, anchor0=-3, rot_stride=-2)
    assert _same(lib, L, 9, 2, 3, p, 1, 3)[1] == 1
    # radial w0 = 0 means the frame size
    pa, pb = OM.MaskParams(block=4, w0=0), OM.MaskParams(block=4, w0=6)
    ka = _same(lib, R, 9, 2, 3, pa, 0, 0)
    assert ka == (OK, 1)
    assert np.array_equal(OM.block_mask_literal(R, 9, 2, 3, pa, 0),
                          OM.block_mask_literal(R, 9, 2, 3, pb, 0))


def test_cache_host_entries(lib):
    h = ctypes.c_void_p()
    assert lib.va_mask_cache_create(0, ctypes.byref(h)) == ERR_INVALID
    assert lib.va_mask_cache_create(4097, ctypes.byref(h)) == ERR_INVALID
    assert lib.va_mask_cache_create(8, None) == ERR_INVALID
    assert lib.va_mask_cache_create(8, ctypes.byref(h)) == OK and h.value
    hits, misses, entries = ctypes.c_int64(-1), ctypes.c_int64(-1), ctypes.c_int(-1)
    assert lib.va_mask_cache_stats(h, ctypes.byref(hits), ctypes.byref(misses),
                                   ctypes.byref(entries)) == OK
    assert (hits.value, misses.value, entries.value) == (0, 0, 0)
    assert lib.va_mask_cache_stats(None, None, None, None) == ERR_INVALID
    assert lib.va_mask_cache_clear(h) == OK
    assert lib.va_mask_cache_clear(None) == ERR_INVALID
    out = ctypes.c_void_p(1)
    cp = _P(128, 0, 1, 0, 0, 1)
    # null cache / params are rejected before any device call
    assert lib.va_mask_cache_get(None, R, 2, 2, 2, ctypes.byref(cp), 0, ctypes.byref(out),
                                 None) == ERR_INVALID
    assert out.value is None
    assert lib.va_mask_cache_get(h, R, 2, 2, 2, None, 0, ctypes.byref(out), None) == ERR_INVALID
    assert lib.va_mask_cache_destroy(h) == OK
    assert lib.va_mask_cache_destroy(None) == OK


def test_same_rejects_bad_arguments(lib):
    cp = _P(128, 0, 1, 0, 0, 1)
    same = ctypes.c_int(7)
    assert lib.va_mask_same(9, 2, 2, 2, ctypes.byref(cp), 0, 1, ctypes.byref(same)) == ERR_INVALID
    assert same.value == 0
    assert lib.va_mask_same(R, 0, 2, 2, ctypes.byref(cp), 0, 1, ctypes.byref(same)) == ERR_INVALID
    assert lib.va_mask_same(R, 2, 2, 2, None, 0, 1, ctypes.byref(same)) == ERR_INVALID
    assert lib.va_mask_same(R, 2, 2, 2, ctypes.byref(cp), 0, 1, None) == ERR_INVALID
    big = _P(1, 0, 1, 0, 0, 1)  # 2^17 blocks of one token
    assert lib.va_mask_same(R, 2, 256, 256, ctypes.byref(big), 0, 1,
                            ctypes.byref(same)) == ERR_UNSUPPORTED
