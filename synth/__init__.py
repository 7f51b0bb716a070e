"""Seeded synthetic inputs shared by the CUDA path and the CPU oracle.

This module holds no attention, mask, clustering or routing arithmetic. It only
draws numbers: counter-based splitmix64 streams (Steele, Lea & Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014), Box-Muller normals,
round-to-nearest-even bf16 quantisation, and the video-shaped Q/K/V recipe:

* Q and K of one head share 8 low-frequency Fourier modes over the (t, h, w)
  latent grid, plus independent N(0, 0.5^2) noise, so that q.k decays with
  spatiotemporal distance (the energy decay the Radial Attention news page
  describes for video diffusion models);
* V ~ N(0, 1);
* the i.i.d. N(0, 1) fp32 recipe of the tiny LVSA check.

Every value is a pure function of (seed, tensor, batch, head, element index),
so any sub-block can be regenerated exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1

# tensor ids of the streams
Q, K, V, MODES, INIT, GRAD = 1, 2, 3, 4, 5, 6


_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def _lib():
    """The C helper (_gen.c), compiled with gcc on first use into _build/."""
    global _LIB
    if _LIB is None:
        src = os.path.join(_HERE, "_gen.c")
        out_dir = os.path.join(_HERE, "_build")
        so = os.path.join(out_dir, "libsynthgen.so")
        if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
            os.makedirs(out_dir, exist_ok=True)
            tmp = so + ".%d.tmp" % os.getpid()
            subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"],
                           check=True)
            os.replace(tmp, so)
        lib = ctypes.CDLL(so)
        f64p = ctypes.POINTER(ctypes.c_double)
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.synth_normals_f32.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                          ctypes.c_double, f32p]
        lib.synth_add_normals_f32.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                              f64p, f32p]
        lib.synth_round_bf16.argtypes = [ctypes.c_int64, f32p]
        _LIB = lib
    return _LIB


def _f32p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def normals_f32(key: int, n: int, std: float = 1.0, base=None) -> np.ndarray:
    """float32(base + std * normals(key, n)) computed by the C helper.

    Equal to the numpy definition below up to the last float64 bit of libm's
    log/cos/sin before the float32 rounding.
    """
    out = np.empty(n, dtype=np.float32)
    if base is None:
        _lib().synth_normals_f32(key, n, 0.0, std, _f32p(out))
    else:
        base = np.ascontiguousarray(base, dtype=np.float64).reshape(-1)
        assert base.size == n
        _lib().synth_add_normals_f32(key, n, std,
                                     base.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                     _f32p(out))
    return out


def round_bf16_(x: np.ndarray) -> np.ndarray:
    """In-place bf16 rounding of a contiguous float32 array (C helper)."""
    assert x.dtype == np.float32 and x.flags.c_contiguous
    _lib().synth_round_bf16(x.size, _f32p(x))
    return x


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function on a uint64 array (in place safe)."""
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def splitmix64_stream(state: int, n: int) -> np.ndarray:
    """The first n outputs of splitmix64 started from `state`.

    Output i is mix(state + (i + 1) * gamma), which is what the sequential
    generator returns on its (i + 1)-th call.
    """
    with np.errstate(over="ignore"):
        ctr = np.arange(1, n + 1, dtype=np.uint64)
        z = np.uint64(state & _MASK64) + ctr * _GAMMA
        return _mix(z)


def stream_key(seed: int, tensor: int, b: int = 0, h: int = 0) -> int:
    """A 64-bit stream key for (seed, tensor, batch, head)."""
    x = (seed & 0xFFFFFFFF) | (tensor << 32) | (b << 40) | (h << 52)
    with np.errstate(over="ignore"):
        return int(_mix(np.array([x & _MASK64], dtype=np.uint64))[0])


def uniforms(key: int, n: int) -> np.ndarray:
    """n uniforms in (0, 1] as float64: ((z >> 11) + 1) * 2^-53."""
    z = splitmix64_stream(key, n)
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normals(key: int, n: int) -> np.ndarray:
    """n standard normals (float64) by Box-Muller on consecutive uniform pairs."""
    m = (n + 1) // 2
    u = uniforms(key, 2 * m)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    a = 2.0 * np.pi * u[1::2]
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(a)
    out[1::2] = r * np.sin(a)
    return out[:n]


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).reshape(x.shape)


def grid_coords(T: int, H: int, W: int):
    """(t, h, w) of every token n = t*H*W + h*W + w (t-major flattening)."""
    n = np.arange(T * H * W, dtype=np.int64)
    return n // (H * W), (n // W) % H, n % W


def fourier_signal(T: int, H: int, W: int, d: int, key: int, n_modes: int = 8) -> np.ndarray:
    """Sum of n_modes low-frequency cosines over the (t, h, w) grid, [N, d] float64.

    Mode m has integer frequencies (f_t, f_h, f_w) uniform in {0, 1, 2}, a
    phase uniform in [0, 2 pi) and an amplitude vector with N(0, 1/8) entries.
    """
    u = uniforms(key, 4 * n_modes)
    freq = np.minimum((u[: 3 * n_modes] * 3.0).astype(np.int64), 2).reshape(n_modes, 3)
    phase = 2.0 * np.pi * u[3 * n_modes:]
    amp = normals(key ^ 0x5DEECE66D, n_modes * d).reshape(n_modes, d) * np.sqrt(1.0 / 8.0)
    t, h, w = grid_coords(T, H, W)
    arg = 2.0 * np.pi * (np.outer(t / T, freq[:, 0]) + np.outer(h / H, freq[:, 1])
                         + np.outer(w / W, freq[:, 2])) + phase[None, :]
    return np.cos(arg) @ amp


def video_qkv(B: int, heads: int, T: int, H: int, W: int, d: int, seed: int,
              dtype: str = "bf16", noise_std: float = 0.5):
    """Video-shaped Q, K, V of shape [B, heads, N, d] as float32 arrays.

    With dtype "bf16" every value is bf16-representable (RNE), so the arrays
    convert to bf16 exactly.
    """
    N = T * H * W
    q = np.empty((B, heads, N, d), dtype=np.float32)
    k = np.empty_like(q)
    v = np.empty_like(q)
    for b in range(B):
        for h in range(heads):
            sig = fourier_signal(T, H, W, d, stream_key(seed, MODES, b, h))
            q[b, h] = normals_f32(stream_key(seed, Q, b, h), N * d, noise_std, sig).reshape(N, d)
            k[b, h] = normals_f32(stream_key(seed, K, b, h), N * d, noise_std, sig).reshape(N, d)
            v[b, h] = normals_f32(stream_key(seed, V, b, h), N * d).reshape(N, d)
    if dtype == "bf16":
        for x in (q, k, v):
            round_bf16_(x)
    return q, k, v


def iid_qkv(B: int, heads: int, N: int, d: int, seed: int, dtype: str = "f32"):
    """I.i.d. N(0, 1) Q, K, V of shape [B, heads, N, d] (float32)."""
    out = []
    for tensor in (Q, K, V):
        x = np.empty((B, heads, N, d), dtype=np.float32)
        for b in range(B):
            for h in range(heads):
                x[b, h] = normals_f32(stream_key(seed, tensor, b, h), N * d).reshape(N, d)
        out.append(round_bf16_(x) if dtype == "bf16" else x)
    return tuple(out)


def upstream_grad(B: int, heads: int, N: int, d: int, seed: int, dtype: str = "bf16",
                  std: float = 1.0) -> np.ndarray:
    """An upstream gradient dL/dO of shape [B, heads, N, d]: i.i.d. N(0, std^2)
    float32, bf16-representable (RNE) when dtype is "bf16"."""
    x = np.empty((B, heads, N, d), dtype=np.float32)
    for b in range(B):
        for h in range(heads):
            x[b, h] = normals_f32(stream_key(seed, GRAD, b, h), N * d, std).reshape(N, d)
    return round_bf16_(x) if dtype == "bf16" else x


def init_indices(B: int, heads: int, N: int, C: int, seed: int, tensor: int = INIT) -> np.ndarray:
    """Seeded initial centroid indices, [B, heads, C] int32.

    For each (b, h): the first C entries of a Durstenfeld (Fisher-Yates)
    shuffle of [0, N): for i < C, j = i + (r_i mod (N - i)), swap a[i], a[j],
    with r_i the i-th splitmix64 output of the (seed, tensor, b, h) stream.
    These are the random numbers the clustering draws; both the CUDA path and
    the oracle take them as input.
    """
    if not (1 <= C <= N):
        raise ValueError("need 1 <= C <= N")
    out = np.empty((B, heads, C), dtype=np.int32)
    for b in range(B):
        for h in range(heads):
            r = splitmix64_stream(stream_key(seed, tensor, b, h), C)
            a = np.arange(N, dtype=np.int64)
            for i in range(C):
                j = i + int(r[i] % np.uint64(N - i))
                a[i], a[j] = a[j], a[i]
            out[b, h] = a[:C]
    return out
