"""The C-ABI library loads and exports every entry point include/va.h declares.

No compute call is made here (no GPU needed); argument validation that
returns before touching the device is checked.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "va.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(?:int|const char\s*\*)\s+(va_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__._build_module().build()
    return ctypes.CDLL(os.path.join(ROOT, "linear_attention_video_fwd_b300", "libva.so"))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("va_mask_build", "va_sparse_attn_fwd", "va_cluster", "va_compensate_route",
                 "va_device_error", "va_mask_free", "va_mask_csr", "va_mask_to_host"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_only_declared_symbols_are_exported():
    import subprocess
    so = os.path.join(ROOT, "linear_attention_video_fwd_b300", "libva.so")
    out = subprocess.run(["nm", "-D", "--defined-only", so], capture_output=True, text=True).stdout
    exported = sorted({ln.split()[-1] for ln in out.splitlines() if " T va_" in ln})
    assert exported == declared_functions()


def test_status_strings_and_version(lib):
    lib.va_status_string.restype = ctypes.c_char_p
    assert lib.va_status_string(0) == b"ok"
    assert lib.va_status_string(-5) == b"device-side wait timed out"
    assert lib.va_version() >= 100


def test_validation_before_device_work(lib):
    # null output handle / params: rejected on the host
    assert lib.va_mask_build(1, 4, 4, 4, None, 0, None, None) == -1
    assert lib.va_sparse_attn_fwd(None, None, None, None, None, None, 1, 1, 1, 128,
                                  ctypes.c_float(1.0), 1, None) == -1
    assert lib.va_set_wait_limit(ctypes.c_int64(10)) == -1
    assert lib.va_set_wait_limit(ctypes.c_int64(4000000000)) == 0


def test_validation_of_the_other_entries(lib):
    # Every entry rejects null pointers on the host, before any CUDA call.
    f, vp = ctypes.c_float, ctypes.c_void_p
    n = None
    assert lib.va_sparse_attn_bwd(n, n, n, n, n, n, n, n, n, n, 1, 1, 1, 128, f(1.0), 1, n) == -1
    assert lib.va_sparse_attn_fwd_host(n, n, n, n, n, n, 1, 1, 1, 128, f(1.0), 1, n) == -1
    assert lib.va_linear_attn_fwd(n, n, n, n, 1, 1, 1, 128, 1, n) == -1
    assert lib.va_mixed_attn_fwd(n, n, n, n, f(0.5), n, 1, 1, 1, 128, f(1.0), 1, n) == -1
    assert lib.va_cluster_from(n, n, 1, 1, 16, 128, 4, 1, 1, n, n, n, n) == -1
    assert lib.va_lipar_prune(n, 1, 2, 3, 4, 16, f(0.5), 1, n, n, n, n, n) == -1
    assert lib.va_lipar_gather(n, n, n, 1, 1, 24, 128, 1, n, n) == -1
    assert lib.va_lipar_restore(n, n, 1, 1, 24, 128, 1, n, n) == -1
    # misaligned device pointers are rejected the same way (never dereferenced)
    odd = vp(0x1001)
    assert lib.va_linear_attn_fwd(odd, odd, odd, odd, 1, 1, 1, 128, 1, n) == -1


def test_python_binding_imports():
    import linear_attention_video_fwd_b300 as va
    assert va.status_string(va.ERR_OOM) == "device allocation failed"


def test_mask_size_limits_are_checked_on_the_host(lib):
    # Grids beyond the documented limits return before any device work, so
    # these calls need no GPU: N >= 2^30 is invalid, more than
    # VA_MASK_MAX_BLOCKS blocks per side is unsupported (the count kernel tests
    # every block pair), for the allocating and the allocation-free build.
    class P(ctypes.Structure):
        _fields_ = [(n, ctypes.c_int32) for n in
                    ("block", "w0", "local", "period", "anchor0", "rot_stride")]

    with open(os.path.join(ROOT, "include", "va.h")) as f:
        max_blocks = int(re.search(r"#define VA_MASK_MAX_BLOCKS (\d+)", f.read()).group(1))
    assert max_blocks == 65536
    out = ctypes.c_void_p(0)
    p1 = P(1, 0, 1, 0, 0, 1)
    assert lib.va_mask_build(1, 1 << 10, 1 << 10, 1 << 10, ctypes.byref(p1), 0,
                             ctypes.byref(out), None) == -1           # N = 2^30
    assert lib.va_mask_build(1, 1, 1, max_blocks + 1, ctypes.byref(p1), 0,
                             ctypes.byref(out), None) == -2           # one block too many
    assert out.value is None
    nnz = ctypes.c_int64(-1)
    fn = lib.va_mask_build_static
    fn.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                   ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p]
    fake = ctypes.c_void_p(0x10000)                  # never dereferenced: rejected first
    assert fn(1, 1, 1, max_blocks + 1, ctypes.byref(p1), 0, fake, fake, 0,
              ctypes.byref(nnz), None) == -2
    assert fn(1, 1 << 10, 1 << 10, 1 << 10, ctypes.byref(p1), 0, fake, fake, 0,
              ctypes.byref(nnz), None) == -1


def test_csr_validator_on_host_arrays():
    # va_csr_validate works on host arrays alone (no device call): the hand-
    # derived tiny LVSA CSR passes, and each way a list can break is rejected.
    import numpy as np
    import linear_attention_video_fwd_b300 as va
    from conftest import read_golden
    g = read_golden("lvsa_tiny_csr.txt")
    rp = np.array([int(x) for x in g[3]], dtype=np.int32)
    col = np.array([int(x) for x in g[5]], dtype=np.int32)
    assert va.csr_validate(rp, col) == va.OK
    bad_rows = rp.copy()
    bad_rows[2] = bad_rows[1] - 1                          # rows run backwards
    assert va.csr_validate(bad_rows, col) == va.ERR_DEVICE
    bad_nnz = rp.copy()
    bad_nnz[-1] -= 1                                       # last offset is not nnz
    assert va.csr_validate(bad_nnz, col) == va.ERR_DEVICE
    out_of_range = col.copy()
    out_of_range[0] = len(rp) - 1                          # column == nqb
    assert va.csr_validate(rp, out_of_range) == va.ERR_DEVICE
    unsorted = col.copy()
    unsorted[[0, 1]] = unsorted[[1, 0]]                    # not ascending within a row
    assert va.csr_validate(rp, unsorted) == va.ERR_DEVICE
    # a row without its diagonal block: fine as a CSR, not for a mask rule
    nodiag_rp = np.array([0, 1, 2], dtype=np.int32)
    nodiag_col = np.array([1, 0], dtype=np.int32)
    assert va.csr_validate(nodiag_rp, nodiag_col, require_diagonal=False) == va.OK
    assert va.csr_validate(nodiag_rp, nodiag_col) == va.ERR_DEVICE
    assert va.csr_validate(np.zeros(1, dtype=np.int32), col) == va.ERR_INVALID   # nqb = 0
