"""ctypes wrapper of the C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY. The oracle is a plain, single-threaded CPU statement of the
ZeRO shard step, used by the tests, by ``__graft_entry__.smoke()`` and by the bench's
CPU-baseline leg to check and time the GPU library. The product package never imports
it, and it shares no code with the product.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(cc: str = "cc") -> str:
    """Compile liboracle.so when a source is newer than it (building runs nothing)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + ".tmp"
    cmd = [cc, "-std=gnu11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class HParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class Scalars(ctypes.Structure):
    _fields_ = [("overflow", ctypes.c_int32), ("skipped", ctypes.c_int32),
                ("step", ctypes.c_int64), ("ss", ctypes.c_double), ("norm", ctypes.c_double),
                ("clip_coef", ctypes.c_double), ("s", ctypes.c_float),
                ("omb1", ctypes.c_float), ("omb2", ctypes.c_float), ("bc1", ctypes.c_float),
                ("bc2", ctypes.c_float), ("decay", ctypes.c_float), ("lr", ctypes.c_float),
                ("beta1", ctypes.c_float), ("beta2", ctypes.c_float), ("eps", ctypes.c_float)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            L.oracle_partition.argtypes = [_I64, _I32, _I32, ctypes.POINTER(_I64),
                                           ctypes.POINTER(_I64)]
            L.oracle_partition.restype = ctypes.c_int
            L.oracle_memory_bytes.argtypes = [_I64, _I32, _I32, _I32]
            L.oracle_memory_bytes.restype = _I64
            L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.oracle_f16_to_f32.restype = ctypes.c_float
            L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
            L.oracle_f32_to_f16.restype = ctypes.c_uint16
            L.oracle_f32_to_f16_array.argtypes = [_P, _P, _I64]
            L.oracle_f16_to_f32_array.argtypes = [_P, _P, _I64]
            L.oracle_reduce.argtypes = [_I32, _P, _I64, _I64, _P]
            L.oracle_stats.argtypes = [_P, _I64, ctypes.POINTER(_I64),
                                       ctypes.POINTER(ctypes.c_uint64),
                                       ctypes.POINTER(ctypes.c_uint64)]
            L.oracle_stats.restype = ctypes.c_int
            L.oracle_scalars_from_stats.argtypes = [_I64, ctypes.c_uint64, ctypes.c_uint64,
                                                    ctypes.c_float, ctypes.c_float,
                                                    ctypes.POINTER(HParams), _I64,
                                                    ctypes.POINTER(Scalars)]
            L.oracle_adam.argtypes = [_I64, _P, _P, _P, _P, _P, ctypes.POINTER(Scalars)]
            L.oracle_step.argtypes = [_I32, _P, _I64, _I64, _P, _P, _P, _P, _P,
                                      ctypes.c_float, ctypes.c_float, ctypes.POINTER(HParams),
                                      _I64, ctypes.POINTER(Scalars)]
            L.oracle_scaler_update.argtypes = [ctypes.POINTER(ctypes.c_float),
                                               ctypes.POINTER(_I32), _I32, ctypes.c_float,
                                               ctypes.c_float, _I32]
            L.oracle_gather.argtypes = [_I32, _I64, _P, _I32, _P, _P]
            L.oracle_gather_source.argtypes = [_I64, _I64, ctypes.POINTER(_I32),
                                               ctypes.POINTER(_I64)]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _ptr_array(arrs) -> ctypes.Array:
    return (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


@dataclass
class Hyper:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01

    def c(self) -> HParams:
        return HParams(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay)


def partition(n: int, nd: int, align: int) -> tuple[int, int]:
    np_, s = _I64(), _I64()
    if lib().oracle_partition(n, nd, align, ctypes.byref(np_), ctypes.byref(s)) != 0:
        raise ValueError("bad partition arguments")
    return np_.value, s.value


def memory_bytes(n: int, nd: int, align: int, stage: int) -> int:
    return lib().oracle_memory_bytes(n, nd, align, stage)


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    lib().oracle_f16_to_f32_array(_ptr(h), _ptr(out), h.size)
    return out


def f32_to_f16(x: np.ndarray) -> np.ndarray:
    """fp16 bit patterns (uint16) of the fp32 input, nearest-even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_f32_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


def reduce(contrib, n_valid: int | None = None) -> np.ndarray:
    """fp32 rank-order sum of the fp16 contributions (uint16 bit patterns)."""
    contrib = [np.ascontiguousarray(c, dtype=np.uint16) for c in contrib]
    n = contrib[0].size
    nv = n if n_valid is None else n_valid
    out = np.empty(n, dtype=np.float32)
    lib().oracle_reduce(len(contrib), _ptr_array(contrib), n, nv, _ptr(out))
    return out


def stats(gsum: np.ndarray) -> tuple[int, int]:
    """(non-finite count, exact sum of (gsum * 2^24)^2 as a Python int)."""
    gsum = np.ascontiguousarray(gsum, dtype=np.float32)
    bad, lo, hi = _I64(), ctypes.c_uint64(), ctypes.c_uint64()
    rc = lib().oracle_stats(_ptr(gsum), gsum.size, ctypes.byref(bad), ctypes.byref(lo),
                            ctypes.byref(hi))
    if rc != 0:
        raise OverflowError("sum of squares exceeds 128 bits")
    return bad.value, (hi.value << 64) | lo.value


def scalars(nonfinite: int, ss_int: int, loss_scale: float, clip: float, hp: Hyper,
            t: int) -> Scalars:
    out = Scalars()
    hpc = hp.c()
    lib().oracle_scalars_from_stats(nonfinite, ss_int & ((1 << 64) - 1), ss_int >> 64,
                                    loss_scale, clip, ctypes.byref(hpc), t, ctypes.byref(out))
    return out


def adam(gsum, master, exp_avg, exp_avg_sq, param16, sc: Scalars) -> None:
    """In-place update of master/exp_avg/exp_avg_sq (float32) and param16 (uint16)."""
    n = gsum.size
    for a, dt in ((gsum, np.float32), (master, np.float32), (exp_avg, np.float32),
                  (exp_avg_sq, np.float32), (param16, np.uint16)):
        assert a.dtype == dt and a.flags["C_CONTIGUOUS"] and a.size == n
    lib().oracle_adam(n, _ptr(gsum), _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
                      _ptr(param16), ctypes.byref(sc))


def step(contrib, master, exp_avg, exp_avg_sq, param16, loss_scale: float, clip: float,
         hp: Hyper, t: int, n_valid: int | None = None) -> Scalars:
    """One shard step over a span, in place. Returns the step's scalars."""
    contrib = [np.ascontiguousarray(c, dtype=np.uint16) for c in contrib]
    n = contrib[0].size
    nv = n if n_valid is None else n_valid
    work = np.empty(n, dtype=np.float32)
    out = Scalars()
    hpc = hp.c()
    for a, dt in ((master, np.float32), (exp_avg, np.float32), (exp_avg_sq, np.float32),
                  (param16, np.uint16)):
        assert a.dtype == dt and a.flags["C_CONTIGUOUS"] and a.size == n
    lib().oracle_step(len(contrib), _ptr_array(contrib), n, nv, _ptr(master), _ptr(exp_avg),
                      _ptr(exp_avg_sq), _ptr(param16), _ptr(work), loss_scale, clip,
                      ctypes.byref(hpc), t, ctypes.byref(out))
    return out


def gather(shards, shard_len: int, layer_offsets) -> list[np.ndarray]:
    shards = [np.ascontiguousarray(s, dtype=np.uint16) for s in shards]
    offs = np.ascontiguousarray(layer_offsets, dtype=np.int64)
    n_layers = offs.size - 1
    dst = [np.zeros(int(offs[l + 1] - offs[l]), dtype=np.uint16) for l in range(n_layers)]
    lib().oracle_gather(len(shards), shard_len, _ptr_array(shards), n_layers, _ptr(offs),
                        _ptr_array(dst))
    return dst


def gather_source(shard_len: int, i: int) -> tuple[int, int]:
    r, off = _I32(), _I64()
    lib().oracle_gather_source(shard_len, i, ctypes.byref(r), ctypes.byref(off))
    return r.value, off.value


def scaler_update(scale: float, good_steps: int, overflow: bool, growth: float = 2.0,
                  backoff: float = 0.5, interval: int = 2000) -> tuple[float, int]:
    """(new fp32 scale, new good-step count) after one step."""
    sc = ctypes.c_float(scale)
    g = _I32(good_steps)
    lib().oracle_scaler_update(ctypes.byref(sc), ctypes.byref(g), 1 if overflow else 0, growth,
                               backoff, interval)
    return sc.value, g.value
