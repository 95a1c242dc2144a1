"""Seeded synthetic inputs for the ZeRO shard step: gradients, master weights, moments.

This module holds no arithmetic of the method itself. It only draws numbers. It is
the one piece that the oracle side and the CUDA side share, and both consume the
bytes it produces as plain inputs.

Definition of the generator (identical on the CPU here and in ``synth.cu`` on the GPU):

* ``mix(z)`` is the SplitMix64 output function (Steele, Lea and Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014): xor-shift 30,
  multiply, xor-shift 27, multiply, xor-shift 31, all modulo 2**64.
* A stream is named by ``(seed, kind, cfg, step, rank)``. Its key is
  ``k = mix(seed + G)`` followed by ``k = mix(k ^ (part + G))`` for each part in
  ``(kind, cfg, step, rank)``, where ``G = 0x9E3779B97F4A7C15``.
* Counter ``c`` of a stream is the 64-bit word ``mix(k + G * (c + 1))``.
* Element ``i`` uses the words for counters ``2i`` and ``2i+1``. Their eight
  16-bit lanes are summed and centred: ``z = sum(lanes) - 4 * 65535``. This is an
  Irwin-Hall(8) variate, a bell-shaped stand-in for a normal that is bounded at
  about 4.9 sigma and needs no transcendental function, so both sides produce
  identical bits.
* The fp32 value is ``float32(z) * c`` where ``c = float32(sigma / sd)`` and
  ``sd = sqrt(8 * (2**32 - 1) / 12)`` is the standard deviation of ``z``. Both
  factors are exact fp32 numbers and the product is one IEEE multiply, rounded to
  nearest even. fp16 outputs round that fp32 value to fp16 (nearest even).
* Elements at flat index ``>= n_valid`` (the partition padding) are 0.

Nothing here depends on the GPU. The device fill lives in ``synth.cu`` and is loaded
on demand by :func:`device_lib`.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

G = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1

# stream kinds
GRAD = 1
MASTER = 2
EXP_AVG = 3
EXP_AVG_SQ = 4
SHARD16 = 5
INJECT = 6

SD_IH8 = math.sqrt(8.0 * (2.0 ** 32 - 1.0) / 12.0)


def mix(z: int) -> int:
    """SplitMix64 output function on one Python int (mod 2**64)."""
    z &= _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def stream_key(seed: int, kind: int, cfg: int, step: int, rank: int) -> int:
    k = mix((seed + G) & _MASK)
    for part in (kind, cfg, step, rank):
        k = mix(k ^ ((part + G) & _MASK))
    return k


def scale_for(sigma: float) -> np.float32:
    """The fp32 factor that maps an Irwin-Hall(8) integer to N(0, sigma)-like values."""
    return np.float32(sigma / SD_IH8)


def _mix_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def ih8(key: int, start: int, n: int) -> np.ndarray:
    """Irwin-Hall(8) integers (as int32) for element indices ``start .. start+n-1``."""
    idx = np.arange(start, start + n, dtype=np.uint64)
    k = np.uint64(key)
    g = np.uint64(G)
    with np.errstate(over="ignore"):
        w0 = _mix_np(k + g * (np.uint64(2) * idx + np.uint64(1)))
        w1 = _mix_np(k + g * (np.uint64(2) * idx + np.uint64(2)))
    s = np.zeros(n, dtype=np.int64)
    m16 = np.uint64(0xFFFF)
    for w in (w0, w1):
        for lane in range(4):
            s += ((w >> np.uint64(16 * lane)) & m16).astype(np.int64)
    return (s - 4 * 65535).astype(np.int32)


def values_f32(key: int, sigma: float, start: int, n: int, n_valid: int | None = None,
               absolute: bool = False) -> np.ndarray:
    z = ih8(key, start, n).astype(np.float32)
    out = z * scale_for(sigma)
    if absolute:
        out = np.abs(out)
    if n_valid is not None:
        idx = np.arange(start, start + n)
        out[idx >= n_valid] = 0.0
    return out.astype(np.float32)


def values_f16(key: int, sigma: float, start: int, n: int, n_valid: int | None = None) -> np.ndarray:
    """fp16 values; returned as uint16 bit patterns."""
    return values_f32(key, sigma, start, n, n_valid).astype(np.float16).view(np.uint16)


def inject_index(seed: int, cfg: int, step: int, rank: int, n: int) -> int:
    """A seeded index in [0, n): the first word of the INJECT stream, modulo n."""
    k = stream_key(seed, INJECT, cfg, step, rank)
    return mix((k + G) & _MASK) % n


# ----------------------------------------------------------------------------------
# device fill (CUDA); compiled from synth.cu into libsynth.so beside this file

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = os.path.join(_HERE, "libsynth.so")
_SRC = os.path.join(_HERE, "synth.cu")
_lock = threading.Lock()
_lib = None


def build(nvcc: str = "nvcc") -> str:
    """Compile libsynth.so for sm_103a when the source is newer than the library."""
    if os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
           "-Xcompiler", "-fPIC", "-shared", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def device_lib():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB):
                raise RuntimeError("libsynth.so is not built; call synth.build()")
            lib = ctypes.CDLL(_LIB)
            lib.synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                                       ctypes.c_float, ctypes.c_int32, ctypes.c_void_p]
            lib.synth_fill.restype = ctypes.c_int
            _lib = lib
    return _lib


F16, F32, F32_ABS = 0, 1, 2


def fill(tensor, key: int, sigma: float, start: int = 0, n_valid: int | None = None,
         stream=None) -> None:
    """Fill a contiguous CUDA tensor (float16 or float32) on its device.

    Element ``j`` of ``tensor`` takes the value of flat index ``start + j``. With
    ``absolute=True`` semantics selected by passing ``sigma < 0``, fp32 values are
    made non-negative (|N(0, |sigma|)|).
    """
    import torch
    assert tensor.is_cuda and tensor.is_contiguous()
    if tensor.dtype == torch.float16:
        mode = F16
    elif tensor.dtype == torch.float32:
        mode = F32_ABS if sigma < 0 else F32
    else:
        raise TypeError("fill supports float16 and float32")
    n = tensor.numel()
    nv = start + n if n_valid is None else n_valid
    c = float(scale_for(abs(sigma)))
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    rc = device_lib().synth_fill(ctypes.c_void_p(tensor.data_ptr()), mode, n, start, nv,
                                 ctypes.c_uint64(key), c, 0, ctypes.c_void_p(s))
    if rc != 0:
        raise RuntimeError(f"synth_fill failed with CUDA error {rc}")
