"""va_mask_build_static: the allocation-free mask build, called through the C ABI.

Some callers cannot allocate device memory on this path: code running under a
caching or arena allocator that owns the whole device, real-time loops where a
cudaMalloc would stall or synchronise the device, embedders whose memory is
handed out by the host framework. For them the library keeps the build's
scratch in a statically sized device array and takes the output arrays from
the caller. This test checks that entry point's CSR against the allocating
va_mask_build (bit-exact, the tolerance every mask test uses) on two calls in
a row, so the shared scratch left by the first call cannot leak into the
second. The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

CASES = [
    # kind, T, H, W, block, w0, local, period, anchor0, rot_stride, step
    (2, 126, 30, 52, 128, 0, 2, 8, 0, 1, 3),   # LVSA long horizon, rotated anchors
    (1, 21, 30, 52, 128, 0, 1, 0, 0, 1, 0),    # Wan-shaped radial
    (1, 9, 4, 4, 32, 3, 1, 0, 0, 1, 0),        # small radial, ragged
]


def _static_fn(va):
    fn = va.lib().va_mask_build_static
    fn.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.POINTER(va._MaskParams), ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_int64, ctypes.POINTER(ctypes.c_int64),
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _outputs(case, capacity):
    """Caller-owned output arrays, filled with garbage to catch unwritten slots."""
    kind, T, H, W, block = case[:5]
    nqb = -(-(T * H * W) // block)
    dev = torch.device("cuda", 0)
    row_ptr = torch.full((nqb + 1,), -7, dtype=torch.int32, device=dev)
    col = torch.full((max(capacity, 1),), -7, dtype=torch.int32, device=dev)
    return row_ptr, col


def _call(va, case, row_ptr, col, capacity):
    kind, T, H, W, block, w0, local, period, a0, rho, step = case
    nnz = ctypes.c_int64(-1)
    p = va._MaskParams(block, w0, local, period, a0, rho)
    stream = torch.cuda.current_stream()
    st = _static_fn(va)(kind, T, H, W, ctypes.byref(p), step,
                        ctypes.c_void_p(row_ptr.data_ptr()), ctypes.c_void_p(col.data_ptr()),
                        capacity, ctypes.byref(nnz), ctypes.c_void_p(stream.cuda_stream))
    torch.cuda.synchronize()
    return st, nnz.value


def _static_build(va, case, capacity):
    row_ptr, col = _outputs(case, capacity)
    st, nnz = _call(va, case, row_ptr, col, capacity)
    return st, nnz, row_ptr.cpu().numpy(), col.cpu().numpy()


def _reference(va, case):
    kind, T, H, W, block, w0, local, period, a0, rho, step = case
    m = va.mask_build(kind, T, H, W, block=block, w0=w0, local=local, period=period,
                      anchor0=a0, rot_stride=rho, step=step)
    rp, col = m.csr()
    m.free()
    return rp, col


def test_static_build_matches_allocating_build_twice_in_a_row(va):
    for case in CASES:
        want_rp, want_col = _reference(va, case)
        for _ in range(2):
            st, nnz, rp, col = _static_build(va, case, len(want_col) + 5)
            assert st == va.OK, va.status_string(st)
            assert nnz == len(want_col)
            assert np.array_equal(rp, want_rp)
            assert np.array_equal(col[:nnz], want_col)
            assert (col[nnz:] == -7).all()            # nothing written past nnz
    assert va.device_error() == va.OK


def test_static_build_reports_size_and_limits(va):
    case = CASES[1]
    want_rp, want_col = _reference(va, case)
    st, nnz, rp, col = _static_build(va, case, 10)            # capacity too small
    assert st == va.ERR_INVALID and nnz == len(want_col)
    assert (col == -7).all()
    st, nnz, _, _ = _static_build(va, (1, 1 << 12, 1 << 6, 1 << 6, 1, 0, 1, 0, 0, 1, 0), 0)
    assert st == va.ERR_UNSUPPORTED                            # beyond the static scratch
    st, nnz, rp, col = _static_build(va, case, len(want_col))  # works again afterwards
    assert st == va.OK and np.array_equal(col[:nnz], want_col)
    assert va.device_error() == va.OK


def test_static_build_allocates_nothing(va, monkeypatch):
    # The property the entry point exists for. (1) With every library scratch
    # allocation made to fail (VA_FAULT_INJECT=alloc), the allocating build
    # fails and the static build still succeeds with the same CSR. (2) Around
    # a warmed-up call (its kernels already loaded), the device's free memory
    # does not move.
    case = CASES[1]
    want_rp, want_col = _reference(va, case)
    row_ptr, col = _outputs(case, len(want_col))
    assert _call(va, case, row_ptr, col, len(want_col)) == (va.OK, len(want_col))
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    monkeypatch.setenv("VA_FAULT_INJECT", "alloc")
    with pytest.raises(va.VAError) as e:
        _reference(va, case)
    assert e.value.status == va.ERR_OOM
    st, nnz = _call(va, case, row_ptr, col, len(want_col))
    monkeypatch.delenv("VA_FAULT_INJECT")
    assert st == va.OK and nnz == len(want_col)
    for _ in range(3):
        assert _call(va, case, row_ptr, col, len(want_col)) == (va.OK, len(want_col))
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before, (free_before, free_after)
    assert np.array_equal(row_ptr.cpu().numpy(), want_rp)
    assert np.array_equal(col.cpu().numpy(), want_col)
    assert va.device_error() == va.OK


def test_static_build_rejects_more_live_pairs_than_int32_offsets(va):
    # The dense mask of 65,536 one-token blocks (the block limit) has 2^32 live
    # block pairs: the count is reported, row_ptr is unusable and col_idx is
    # left untouched.
    case = (0, 1, 1, 65536, 1, 0, 1, 0, 0, 1, 0)
    st, nnz, _, col = _static_build(va, case, 16)
    assert st == va.ERR_UNSUPPORTED and nnz == 1 << 32
    assert (col == -7).all()
    assert va.device_error() == va.OK


def test_python_wrapper_two_phase(va):
    # size query with an empty col_idx, then the build into an exact array
    kind, T, H, W, block, w0, local, period, a0, rho, step = CASES[2]
    kw = dict(block=block, w0=w0, local=local, period=period, anchor0=a0, rot_stride=rho,
              step=step)
    nqb = -(-(T * H * W) // block)
    dev = torch.device("cuda", 0)
    row_ptr = torch.empty(nqb + 1, dtype=torch.int32, device=dev)
    with pytest.raises(va.VAError) as e:
        va.mask_build_static(kind, T, H, W, row_ptr,
                             torch.empty(0, dtype=torch.int32, device=dev), **kw)
    need = e.value.nnz
    assert need > 0
    col = torch.empty(need, dtype=torch.int32, device=dev)
    assert va.mask_build_static(kind, T, H, W, row_ptr, col, **kw) == need
    torch.cuda.synchronize()
    m = va.mask_build(kind, T, H, W, **kw)
    rp, cl = m.csr()
    assert np.array_equal(row_ptr.cpu().numpy(), rp) and np.array_equal(col.cpu().numpy(), cl)
    m.free()
    with pytest.raises(va.VAError):  # a short row_ptr is refused on the host
        va.mask_build_static(kind, T, H, W, row_ptr[:nqb], col, **kw)
    assert va.device_error() == va.OK
