"""Block-sparse video attention for NVIDIA B300 (sm_103a).

Thin Python binding over the C ABI in ``include/va.h`` (``libva.so``, built
in-tree by ``build.py``). Every operation runs in the library's CUDA kernels;
this module only marshals torch tensors (device memory) and the current CUDA
stream into the C calls. There is no CPU implementation here: if ``libva.so``
is missing, importing the binding raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libva.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_OOM, ERR_TIMEOUT, ERR_DEVICE = 0, -1, -2, -3, -4, -5, -6
DENSE, RADIAL, LVSA = 0, 1, 2
F32, BF16 = 0, 1


class VAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed: %s (%d)" % (what, status_string(status), status))
        self.status = status


class _MaskParams(ctypes.Structure):
    _fields_ = [("block", ctypes.c_int32), ("w0", ctypes.c_int32), ("local", ctypes.c_int32),
                ("period", ctypes.c_int32), ("anchor0", ctypes.c_int32),
                ("rot_stride", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libva.so is not built (%s); run __graft_entry__.build() or "
                          "python linear_attention_video_fwd_b300/build.py" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, f64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                              ctypes.c_double)
    i32p = ctypes.POINTER(ctypes.c_int32)
    sig = {
        "va_mask_build": [i32, i32, i32, i32, ctypes.POINTER(_MaskParams), i32,
                          ctypes.POINTER(vp), vp],
        "va_mask_csr": [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i32),
                        ctypes.POINTER(i64)],
        "va_mask_info": [vp, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i64)],
        "va_mask_to_host": [vp, i32p, i32p],
        "va_mask_free": [vp],
        "va_mask_build_static": [i32, i32, i32, i32, ctypes.POINTER(_MaskParams), i32, vp, vp,
                                 i64, ctypes.POINTER(i64), vp],
        "va_mask_cache_create": [i32, ctypes.POINTER(vp)],
        "va_mask_cache_get": [vp, i32, i32, i32, i32, ctypes.POINTER(_MaskParams), i32,
                              ctypes.POINTER(vp), vp],
        "va_mask_cache_stats": [vp, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                ctypes.POINTER(i32)],
        "va_mask_cache_clear": [vp],
        "va_mask_cache_destroy": [vp],
        "va_mask_same": [i32, i32, i32, i32, ctypes.POINTER(_MaskParams), i32, i32,
                         ctypes.POINTER(i32)],
        "va_sparse_attn_fwd": [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp],
        "va_sparse_attn_fwd_host": [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp],
        "va_sparse_attn_bwd": [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32,
                               i32, vp],
        "va_linear_attn_fwd": [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp],
        "va_mixed_attn_fwd": [vp, vp, vp, vp, f32, vp, i32, i32, i32, i32, f32, i32, vp],
        "va_cluster": [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp],
        "va_cluster_from": [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp],
        "va_lipar_prune": [vp, i32, i32, i32, i32, i32, f32, i32, vp, vp, vp, vp, vp],
        "va_lipar_gather": [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp],
        "va_lipar_restore": [vp, vp, i32, i32, i32, i32, i32, vp, vp],
        "va_compensate_route": [vp, vp, vp, vp, i32, vp, i32, f64, f32, i32, i32, i32, i32, i32,
                                vp, vp, vp, vp],
        "va_device_error": [vp],
        "va_set_wait_limit": [i64],
        "va_selftest_wait_timeout": [i64, vp],
        "va_csr_validate": [i32p, i32p, i32, i64, i32],
        "va_status_string": [i32],
        "va_version": [],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "va_status_string" else ctypes.c_int
    return lib


_lib = _load()


def lib():
    """The loaded ctypes library (C ABI of include/va.h)."""
    return _lib


def status_string(status: int) -> str:
    return _lib.va_status_string(status).decode()


def _check(status: int, what: str):
    if status != OK:
        raise VAError(status, what)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise VAError(ERR_UNSUPPORTED, "dtype %s" % t.dtype)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise VAError(ERR_INVALID, "tensor argument (needs contiguous CUDA tensors)")


class Mask:
    """A library-owned block mask (device CSR). Free with .free() or on GC;
    a mask from a MaskCache belongs to the cache and is freed by it."""

    def __init__(self, handle, kind, T, H, W, params, step, cache=None):
        self._h = handle
        self._cache = cache
        self._gen = cache._gen if cache is not None else 0
        self.kind, self.T, self.H, self.W, self.step = kind, T, H, W, step
        self.params = params
        nqb, nnz = ctypes.c_int(), ctypes.c_int64()
        _check(_lib.va_mask_csr(self._h, None, None, ctypes.byref(nqb), ctypes.byref(nnz)),
               "va_mask_csr")
        N, block, lp = ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
        _check(_lib.va_mask_info(self._h, ctypes.byref(N), ctypes.byref(block), ctypes.byref(lp)),
               "va_mask_info")
        self.nqb, self.nnz, self.N, self.block, self.live_pairs = (
            nqb.value, nnz.value, N.value, block.value, lp.value)

    @property
    def handle(self):
        c = self._cache
        if c is not None and (c._h is None or c._gen != self._gen):
            raise VAError(ERR_INVALID, "mask of a cleared or closed MaskCache")
        return self._h

    def csr(self):
        """(row_ptr [nqb+1], col_idx [nnz]) as host int32 arrays."""
        rp = np.zeros(self.nqb + 1, dtype=np.int32)
        col = np.zeros(max(self.nnz, 1), dtype=np.int32)
        _check(_lib.va_mask_to_host(self._h, rp.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                    col.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
               "va_mask_to_host")
        return rp, col[: self.nnz]

    def free(self):
        if self._h and self._cache is None:
            _lib.va_mask_free(self._h)
        self._h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def mask_build(kind: int, T: int, H: int, W: int, block: int = 128, w0: int = 0, local: int = 1,
               period: int = 0, anchor0: int = 0, rot_stride: int = 1, step: int = 0,
               stream=None) -> Mask:
    """va_mask_build: the static block mask of a T x H x W latent grid."""
    p = _MaskParams(block, w0, local, period, anchor0, rot_stride)
    h = ctypes.c_void_p()
    _check(_lib.va_mask_build(kind, T, H, W, ctypes.byref(p), step, ctypes.byref(h),
                              _stream(stream)), "va_mask_build")
    return Mask(h, kind, T, H, W, p, step)


def mask_build_static(kind: int, T: int, H: int, W: int, row_ptr, col_idx, block: int = 128,
                      w0: int = 0, local: int = 1, period: int = 0, anchor0: int = 0,
                      rot_stride: int = 1, step: int = 0, stream=None) -> int:
    """va_mask_build_static: the mask's CSR written into caller-owned int32 CUDA
    tensors row_ptr [nqb + 1] and col_idx [capacity], with no device allocation.
    Returns nnz. If col_idx is too small, raises VAError with .nnz set to the
    length needed (col_idx untouched)."""
    import torch
    _require_cuda(row_ptr, col_idx)
    if row_ptr.dtype != torch.int32 or col_idx.dtype != torch.int32:
        raise VAError(ERR_INVALID, "row_ptr / col_idx dtype (needs int32)")
    nqb = -(-(T * H * W) // block) if block > 0 else 0
    if row_ptr.numel() < nqb + 1:
        raise VAError(ERR_INVALID, "row_ptr length (needs nqb + 1 = %d)" % (nqb + 1))
    p = _MaskParams(block, w0, local, period, anchor0, rot_stride)
    nnz = ctypes.c_int64(-1)
    cap = col_idx.numel()
    st = _lib.va_mask_build_static(kind, T, H, W, ctypes.byref(p), step, _ptr(row_ptr),
                                   _ptr(col_idx if cap > 0 else None), cap, ctypes.byref(nnz),
                                   _stream(stream))
    if st != OK:
        e = VAError(st, "va_mask_build_static")
        e.nnz = nnz.value
        raise e
    return nnz.value


def version() -> int:
    """va_version: the library's version number."""
    return _lib.va_version()


def _mask_params(block, w0, local, period, anchor0, rot_stride):
    return _MaskParams(block, w0, local, period, anchor0, rot_stride)


class MaskCache:
    """va_mask_cache: block masks reused across denoising steps. get() builds a
    mask on its first request and returns the cached one afterwards; requests
    that differ only in what the CSR does not depend on (the step of a radial
    mask, the LVSA rotation phase) share one entry."""

    def __init__(self, capacity: int = 64):
        h = ctypes.c_void_p()
        _check(_lib.va_mask_cache_create(capacity, ctypes.byref(h)), "va_mask_cache_create")
        self._h = h
        self._gen = 0

    def get(self, kind: int, T: int, H: int, W: int, block: int = 128, w0: int = 0,
            local: int = 1, period: int = 0, anchor0: int = 0, rot_stride: int = 1,
            step: int = 0, stream=None) -> Mask:
        if self._h is None:
            raise VAError(ERR_INVALID, "closed MaskCache")
        p = _mask_params(block, w0, local, period, anchor0, rot_stride)
        m = ctypes.c_void_p()
        _check(_lib.va_mask_cache_get(self._h, kind, T, H, W, ctypes.byref(p), step,
                                      ctypes.byref(m), _stream(stream)), "va_mask_cache_get")
        return Mask(m, kind, T, H, W, p, step, cache=self)

    def stats(self):
        """(hits, misses, entries)."""
        hits, misses, entries = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int()
        _check(_lib.va_mask_cache_stats(self._h, ctypes.byref(hits), ctypes.byref(misses),
                                        ctypes.byref(entries)), "va_mask_cache_stats")
        return hits.value, misses.value, entries.value

    def clear(self):
        """Free every cached mask; masks returned earlier become invalid."""
        self._gen += 1
        _check(_lib.va_mask_cache_clear(self._h), "va_mask_cache_clear")

    def close(self):
        if self._h is not None:
            _lib.va_mask_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mask_same(kind: int, T: int, H: int, W: int, step_a: int, step_b: int, block: int = 128,
              w0: int = 0, local: int = 1, period: int = 0, anchor0: int = 0,
              rot_stride: int = 1) -> bool:
    """va_mask_same (host only): whether a MaskCache serves the two steps from
    one entry."""
    p = _mask_params(block, w0, local, period, anchor0, rot_stride)
    same = ctypes.c_int()
    _check(_lib.va_mask_same(kind, T, H, W, ctypes.byref(p), step_a, step_b,
                             ctypes.byref(same)), "va_mask_same")
    return bool(same.value)


def sparse_attn_fwd(q, k, v, mask: Mask, scale: float | None = None, out=None, lse=None,
                    stream=None):
    """va_sparse_attn_fwd on [B, heads, N, d] CUDA tensors. Returns (out, lse or None)."""
    import torch
    _require_cuda(q, k, v, out, lse)
    B, Hh, N, d = q.shape
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise VAError(ERR_INVALID, "q/k/v shapes or dtypes differ")
    if out is None:
        out = torch.empty_like(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(_lib.va_sparse_attn_fwd(_ptr(q), _ptr(k), _ptr(v), mask.handle, _ptr(out), _ptr(lse),
                                   B, Hh, N, d, float(scale), _dtype_code(q), _stream(stream)),
           "va_sparse_attn_fwd")
    return out, lse


def sparse_attn_bwd(q, k, v, out, dout, lse, mask: Mask, scale: float | None = None, dq=None,
                    dk=None, dv=None, stream=None):
    """va_sparse_attn_bwd on [B, heads, N, d] CUDA tensors: the gradients of
    sparse_attn_fwd's output (out, lse from the forward call) for the upstream
    gradient dout. Returns (dq, dk, dv)."""
    import torch
    _require_cuda(q, k, v, out, dout, lse, dq, dk, dv)
    B, Hh, N, d = q.shape
    for t in (k, v, out, dout):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise VAError(ERR_INVALID, "q/k/v/out/dout shapes or dtypes differ")
    if lse is None or lse.shape != (B, Hh, N) or lse.dtype != torch.float32:
        raise VAError(ERR_INVALID, "lse must be float32 [B, heads, N]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(_lib.va_sparse_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                   mask.handle, _ptr(dq), _ptr(dk), _ptr(dv), B, Hh, N, d,
                                   float(scale), _dtype_code(q), _stream(stream)),
           "va_sparse_attn_bwd")
    return dq, dk, dv


def sparse_attn_fwd_host(q, k, v, mask: Mask, scale: float | None = None, out=None, lse=None,
                         stream=None):
    """va_sparse_attn_fwd_host on [B, heads, N, d] CPU tensors (pin them for overlapped
    copies). Asynchronous on `stream` (default: the current CUDA stream): synchronise
    it before reading out / lse. Returns (out, lse or None)."""
    import torch
    for t in (q, k, v, out, lse):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise VAError(ERR_INVALID, "tensor argument (needs contiguous CPU tensors)")
    B, Hh, N, d = q.shape
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise VAError(ERR_INVALID, "q/k/v shapes or dtypes differ")
    if out is None:
        out = torch.empty_like(q, pin_memory=q.is_pinned())
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(_lib.va_sparse_attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), mask.handle, _ptr(out),
                                        _ptr(lse), B, Hh, N, d, float(scale), _dtype_code(q),
                                        _stream(stream)),
           "va_sparse_attn_fwd_host")
    return out, lse


def linear_attn_fwd(q, k, v, out=None, stream=None):
    """va_linear_attn_fwd on [B, heads, N, d] CUDA tensors. Returns out."""
    import torch
    _require_cuda(q, k, v, out)
    B, Hh, N, d = q.shape
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise VAError(ERR_INVALID, "q/k/v shapes or dtypes differ")
    if out is None:
        out = torch.empty_like(q)
    _check(_lib.va_linear_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hh, N, d,
                                   _dtype_code(q), _stream(stream)),
           "va_linear_attn_fwd")
    return out


def mixed_attn_fwd(q, k, v, mask: Mask, r: float, scale: float | None = None, out=None,
                   stream=None):
    """va_mixed_attn_fwd: r * block-sparse attention + (1 - r) * linear attention."""
    import torch
    _require_cuda(q, k, v, out)
    B, Hh, N, d = q.shape
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise VAError(ERR_INVALID, "q/k/v shapes or dtypes differ")
    if out is None:
        out = torch.empty_like(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(_lib.va_mixed_attn_fwd(_ptr(q), _ptr(k), _ptr(v), mask.handle, float(r), _ptr(out), B,
                                  Hh, N, d, float(scale), _dtype_code(q), _stream(stream)),
           "va_mixed_attn_fwd")
    return out


def cluster(x, C: int, iters: int, init_idx, assign=None, centroid=None, count=None,
            stream=None):
    """va_cluster: Lloyd k-means per (batch, head). Returns (assign, centroid, count)."""
    import torch
    _require_cuda(x, init_idx, assign, centroid, count)
    B, Hh, N, d = x.shape
    if init_idx.dtype != torch.int32 or tuple(init_idx.shape) != (B, Hh, C):
        raise VAError(ERR_INVALID, "init_idx must be int32 [B, heads, C]")
    dev = x.device
    if assign is None:
        assign = torch.empty((B, Hh, N), dtype=torch.int32, device=dev)
    if centroid is None:
        centroid = torch.empty((B, Hh, C, d), dtype=torch.float32, device=dev)
    if count is None:
        count = torch.empty((B, Hh, C), dtype=torch.int32, device=dev)
    _check(_lib.va_cluster(_ptr(x), _ptr(init_idx), B, Hh, N, d, C, iters, _dtype_code(x),
                           _ptr(assign), _ptr(centroid), _ptr(count), _stream(stream)),
           "va_cluster")
    return assign, centroid, count


def cluster_from(x, centroid_init, iters: int, assign=None, centroid=None, count=None,
                 stream=None):
    """va_cluster_from: Lloyd k-means warm-started from float32 centroids
    [B, heads, C, d] (may be passed again as `centroid`). Returns (assign, centroid, count)."""
    import torch
    _require_cuda(x, centroid_init, assign, centroid, count)
    B, Hh, N, d = x.shape
    if centroid_init.dtype != torch.float32 or centroid_init.dim() != 4 or \
            tuple(centroid_init.shape[:2]) != (B, Hh) or centroid_init.shape[3] != d:
        raise VAError(ERR_INVALID, "centroid_init must be float32 [B, heads, C, d]")
    C = centroid_init.shape[2]
    dev = x.device
    if assign is None:
        assign = torch.empty((B, Hh, N), dtype=torch.int32, device=dev)
    if centroid is None:
        centroid = torch.empty((B, Hh, C, d), dtype=torch.float32, device=dev)
    if count is None:
        count = torch.empty((B, Hh, C), dtype=torch.int32, device=dev)
    _check(_lib.va_cluster_from(_ptr(x), _ptr(centroid_init), B, Hh, N, d, C, iters,
                                _dtype_code(x), _ptr(assign), _ptr(centroid), _ptr(count),
                                _stream(stream)),
           "va_cluster_from")
    return assign, centroid, count


def lipar_prune(x, T: int, H: int, W: int, tau: float, stream=None):
    """va_lipar_prune on a [B, T*H*W, C] CUDA latent.
    Returns (keep uint8 [B, N], order int32 [B, N], src int32 [B, N], count int32 [B])."""
    import torch
    _require_cuda(x)
    B, N, C = x.shape
    if N != T * H * W:
        raise VAError(ERR_INVALID, "x must be [B, T*H*W, C]")
    dev = x.device
    keep = torch.empty((B, N), dtype=torch.uint8, device=dev)
    order = torch.empty((B, N), dtype=torch.int32, device=dev)
    src = torch.empty((B, N), dtype=torch.int32, device=dev)
    count = torch.empty((B,), dtype=torch.int32, device=dev)
    _check(_lib.va_lipar_prune(_ptr(x), B, T, H, W, C, float(tau), _dtype_code(x), _ptr(keep),
                               _ptr(order), _ptr(src), _ptr(count), _stream(stream)),
           "va_lipar_prune")
    return keep, order, src, count


def lipar_gather(x, order, count, out=None, stream=None):
    """va_lipar_gather: compacted copy of a [B, heads, N, d] CUDA tensor."""
    import torch
    _require_cuda(x, order, count, out)
    B, Hh, N, d = x.shape
    if out is None:
        out = torch.zeros_like(x)
    _check(_lib.va_lipar_gather(_ptr(x), _ptr(order), _ptr(count), B, Hh, N, d, _dtype_code(x),
                                _ptr(out), _stream(stream)),
           "va_lipar_gather")
    return out


def lipar_restore(y, src, out=None, stream=None):
    """va_lipar_restore: full-length [B, heads, N, d] result from a compacted one."""
    import torch
    _require_cuda(y, src, out)
    B, Hh, N, d = y.shape
    if out is None:
        out = torch.empty_like(y)
    _check(_lib.va_lipar_restore(_ptr(y), _ptr(src), B, Hh, N, d, _dtype_code(y), _ptr(out),
                                 _stream(stream)),
           "va_lipar_restore")
    return out


def compensate_route(q, k, v, qassign, Cq: int, kassign, Ck: int, density: float,
                     scale: float | None = None, out=None, err=None, sel=None, stream=None):
    """va_compensate_route. Returns (out, err or None, sel or None)."""
    import torch
    _require_cuda(q, k, v, qassign, kassign, out, err, sel)
    B, Hh, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(_lib.va_compensate_route(_ptr(q), _ptr(k), _ptr(v), _ptr(qassign), Cq, _ptr(kassign),
                                    Ck, float(density), float(scale), B, Hh, N, d,
                                    _dtype_code(q), _ptr(out), _ptr(err), _ptr(sel),
                                    _stream(stream)), "va_compensate_route")
    return out, err, sel


def csr_validate(row_ptr, col_idx, require_diagonal: bool = True) -> int:
    """va_csr_validate on host int32 arrays: VA_OK, ERR_DEVICE or ERR_INVALID."""
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    col = np.ascontiguousarray(col_idx, dtype=np.int32)
    p32 = ctypes.POINTER(ctypes.c_int32)
    return _lib.va_csr_validate(rp.ctypes.data_as(p32), col.ctypes.data_as(p32), len(rp) - 1,
                                len(col), 1 if require_diagonal else 0)


def device_error(stream=None) -> int:
    """va_device_error: sync the stream and return/clear the device error word."""
    return _lib.va_device_error(_stream(stream))


def selftest_wait_timeout(cycles: int = 2_000_000, stream=None):
    """va_selftest_wait_timeout: a bounded device wait that must give up."""
    _check(_lib.va_selftest_wait_timeout(int(cycles), _stream(stream)), "va_selftest_wait_timeout")


def set_wait_limit(cycles: int):
    _check(_lib.va_set_wait_limit(int(cycles)), "va_set_wait_limit")
