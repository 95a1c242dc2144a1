"""Python binding of libzero, the GB300 ZeRO shard-step library (include/zero.h).

Argument marshalling only: every step of the path runs in the library's CUDA kernels.
Functions carry the C names; they accept torch tensors (their ``data_ptr()`` is passed)
or raw integer addresses, and raise :class:`ZeroError` on a non-zero return code.
The first call loads ``libzero.so`` and raises if it has not been built
(``python -m sharded_emulated_reduce_gb300.build``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzero.so")

ZERO_OK = 0
ZERO_EINVAL = -1
ZERO_EALIGN = -2
ZERO_EUNBOUND = -3
ZERO_ECUDA = -4
ZERO_EDEVICE = -5
ZERO_MAX_ND = 256
ZERO_STATS_WORDS = 8
ZERO_PROF_KINDS = 4
ZERO_NOALLOC_MAX_SPAN = 4194304
PROF_REDUCE, PROF_UPDATE, PROF_FINALIZE, PROF_GATHER = range(4)


class ZeroError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"libzero error {code}: {message}")
        self.code = code


class zero_adam_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class zero_step_info(ctypes.Structure):
    _fields_ = [("overflow", ctypes.c_int32), ("skipped", ctypes.c_int32),
                ("status", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("step", ctypes.c_int64), ("global_norm", ctypes.c_double),
                ("sum_sq", ctypes.c_double), ("clip_coef", ctypes.c_double),
                ("scale", ctypes.c_float), ("bc1", ctypes.c_float), ("bc2", ctypes.c_float),
                ("reserved2", ctypes.c_float)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_ if not k.startswith("reserved")}


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F = ctypes.c_float
_PP = ctypes.POINTER(ctypes.c_void_p)

_SIGS = {
    "zero_plan_create": ([_I64, _I32, _I32, _I32, ctypes.POINTER(zero_adam_hparams),
                          ctypes.POINTER(_P)], ctypes.c_int),
    "zero_plan_destroy": ([_P], None),
    "zero_plan_layout": ([_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64)], ctypes.c_int),
    "zero_workspace_bytes": ([_P, _I32, _I32], _I64),
    "zero_plan_bind": ([_P, _I32, _I32, _P, _P, _P, _P, _P, _I64], ctypes.c_int),
    "zero_shard_step": ([_P, _I32, _I32, _PP, _F, _F, _P], ctypes.c_int),
    "zero_shard_reduce": ([_P, _I32, _I32, _PP, _P], ctypes.c_int),
    "zero_shard_stats": ([_P, ctypes.POINTER(_P)], ctypes.c_int),
    "zero_shard_update": ([_P, _I32, _I32, _F, _F, _P], ctypes.c_int),
    "zero_step_result": ([_P, ctypes.POINTER(zero_step_info)], ctypes.c_int),
    "zero_gather_layers": ([_P, ctypes.POINTER(_I64), _I32, _PP, _PP, _P], ctypes.c_int),
    "zero_memory_bytes": ([_I64, _I32, _I32, _I32, ctypes.POINTER(_I64)], ctypes.c_int),
    "zero_profile_enable": ([_P, _I32], ctypes.c_int),
    "zero_profile_read": ([_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I64), _I32],
                          ctypes.c_int),
    "zero_shard_step_noalloc": ([_I32, _I64, _I64, _PP, _P, _P, _P, _P, _P,
                                 ctypes.POINTER(zero_adam_hparams), _F, _F, _P], ctypes.c_int),
    "zero_last_error": ([], ctypes.c_char_p),
}
_lib_handle = None


def lib() -> ctypes.CDLL:
    """The loaded libzero.so. Raises if it has not been built: there is no fallback."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m sharded_emulated_reduce_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _lib_handle = handle
    return _lib_handle


class _Lazy:
    def __getattr__(self, name):
        return getattr(lib(), name)


_lib = _Lazy()

EXPORTED = tuple(_SIGS)


def zero_last_error() -> str:
    return _lib.zero_last_error().decode()


def _check(rc: int) -> int:
    if rc < 0:
        raise ZeroError(rc, zero_last_error())
    return rc


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _ptrs(xs: Sequence) -> ctypes.Array:
    return (ctypes.c_void_p * len(xs))(*[_addr(x) for x in xs])


def _stream(stream) -> int:
    if stream is None:
        import torch
        if torch.cuda.is_available() and torch.cuda.is_initialized():
            return torch.cuda.current_stream().cuda_stream
        return 0
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owner of a ``zero_plan*``; keeps the bound buffers alive while bound."""

    def __init__(self, handle: int, n_params: int, nd: int, stage: int, align: int):
        self.handle = handle
        self.n_params, self.nd, self.stage, self.align = n_params, nd, stage, align
        self._keep = ()

    @property
    def _as_parameter_(self):
        if not self.handle:
            raise ZeroError(ZERO_EINVAL, "plan was destroyed")
        return ctypes.c_void_p(self.handle)

    def close(self) -> None:
        if self.handle:
            _lib.zero_plan_destroy(ctypes.c_void_p(self.handle))
            self.handle = 0
            self._keep = ()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def zero_plan_create(n_params: int, nd: int, stage: int, align: int,
                     hp: zero_adam_hparams | dict) -> Plan:
    if isinstance(hp, dict):
        hp = zero_adam_hparams(**hp)
    out = ctypes.c_void_p()
    _check(_lib.zero_plan_create(n_params, nd, stage, align, ctypes.byref(hp), ctypes.byref(out)))
    return Plan(out.value, n_params, nd, stage, align)


def zero_plan_destroy(plan: Plan) -> None:
    plan.close()


def zero_plan_layout(plan: Plan) -> tuple[int, int]:
    np_, s = _I64(), _I64()
    _check(_lib.zero_plan_layout(plan, ctypes.byref(np_), ctypes.byref(s)))
    return np_.value, s.value


def zero_workspace_bytes(plan: Plan, r0: int, r1: int) -> int:
    return _check(_lib.zero_workspace_bytes(plan, r0, r1))


def zero_plan_bind(plan: Plan, r0: int, r1: int, master, exp_avg, exp_avg_sq, param16,
                   workspace, initial_step: int = 0) -> None:
    _check(_lib.zero_plan_bind(plan, r0, r1, _addr(master), _addr(exp_avg), _addr(exp_avg_sq),
                               _addr(param16), _addr(workspace), initial_step))
    plan._keep = (master, exp_avg, exp_avg_sq, param16, workspace)


def zero_shard_step(plan: Plan, r0: int, r1: int, grads: Sequence, loss_scale: float,
                    clip: float, stream=None) -> None:
    _check(_lib.zero_shard_step(plan, r0, r1, _ptrs(grads), loss_scale, clip, _stream(stream)))


def zero_shard_reduce(plan: Plan, r0: int, r1: int, grads: Sequence, stream=None) -> None:
    _check(_lib.zero_shard_reduce(plan, r0, r1, _ptrs(grads), _stream(stream)))


def zero_shard_stats(plan: Plan) -> int:
    """Device address of the plan's ZERO_STATS_WORDS int64 exchange buffer."""
    p = ctypes.c_void_p()
    _check(_lib.zero_shard_stats(plan, ctypes.byref(p)))
    return p.value


def zero_shard_update(plan: Plan, r0: int, r1: int, loss_scale: float, clip: float,
                      stream=None) -> None:
    _check(_lib.zero_shard_update(plan, r0, r1, loss_scale, clip, _stream(stream)))


def zero_step_result(plan: Plan) -> zero_step_info:
    info = zero_step_info()
    _check(_lib.zero_step_result(plan, ctypes.byref(info)))
    return info


def zero_gather_layers(plan: Plan, layer_offsets: Sequence[int], shards: Sequence,
                       layer_dst: Sequence, stream=None) -> None:
    n_layers = len(layer_offsets) - 1
    offs = (_I64 * len(layer_offsets))(*[int(x) for x in layer_offsets])
    _check(_lib.zero_gather_layers(plan, offs, n_layers, _ptrs(shards), _ptrs(layer_dst),
                                   _stream(stream)))


def zero_memory_bytes(n_params: int, nd: int, align: int, stage: int) -> int:
    out = _I64()
    _check(_lib.zero_memory_bytes(n_params, nd, align, stage, ctypes.byref(out)))
    return out.value


def zero_profile_enable(plan: Plan, on: bool = True) -> None:
    _check(_lib.zero_profile_enable(plan, 1 if on else 0))


def zero_profile_read(plan: Plan, reset: bool = False) -> tuple[list[float], list[int]]:
    ms = (ctypes.c_double * ZERO_PROF_KINDS)()
    n = (_I64 * ZERO_PROF_KINDS)()
    _check(_lib.zero_profile_read(plan, ms, n, 1 if reset else 0))
    return list(ms), list(n)


# ------------------------------------------------------------------------------------
# Spans split across processes (one process per GPU)

def rank_ranges(nd: int, world: int) -> list[tuple[int, int]]:
    """The logical-rank span [r0, r1) of each of ``world`` processes: contiguous, equal
    sized, in process order. ``world`` must divide ``nd``."""
    if world < 1 or nd % world:
        raise ValueError(f"world size {world} must divide Nd = {nd}")
    per = nd // world
    return [(g * per, (g + 1) * per) for g in range(world)]


def stats_words(nonfinite: int, sum_sq: int) -> list[int]:
    """Host view of the exchange-buffer format (zero_shard_stats): word 0 the non-finite
    count, words 1..4 the 32-bit limbs of the exact sum of squares of (gsum * 2^24),
    least significant first, words 5..7 zero."""
    return [nonfinite] + [(sum_sq >> (32 * i)) & 0xFFFFFFFF for i in range(4)] + [0, 0, 0]


def stats_decode(words: Sequence[int]) -> tuple[int, int]:
    """(non-finite count, exact sum of squares) of a (possibly summed) exchange buffer."""
    return int(words[0]), sum(int(words[1 + i]) << (32 * i) for i in range(4))


class _DeviceWords:
    """__cuda_array_interface__ over the plan's device statistics words."""

    def __init__(self, addr: int):
        self.__cuda_array_interface__ = {"shape": (ZERO_STATS_WORDS,), "typestr": "<i8",
                                         "data": (addr, False), "version": 3, "strides": None}


def stats_tensor(plan: Plan):
    """A torch int64 tensor aliasing the plan's exchange buffer on its device."""
    import torch
    return torch.as_tensor(_DeviceWords(zero_shard_stats(plan)), device="cuda")


def zero_dist_step(plan: Plan, r0: int, r1: int, grads: Sequence, loss_scale: float,
                   clip: float, group=None, stream=None) -> None:
    """One shard step of a span split across the processes of a torch.distributed group:
    zero_shard_reduce, an integer sum all-reduce of the statistics words (the exchange
    step; exact, so the result does not depend on the reduction order), then
    zero_shard_update. Every process calls it with its own span."""
    import torch
    import torch.distributed as dist
    s = torch.cuda.current_stream() if stream is None else stream
    zero_shard_reduce(plan, r0, r1, grads, s)
    words = stats_tensor(plan)
    with torch.cuda.stream(s):
        dist.all_reduce(words, op=dist.ReduceOp.SUM, group=group)
    zero_shard_update(plan, r0, r1, loss_scale, clip, s)


def zero_shard_step_noalloc(nd: int, n: int, n_valid: int, grads: Sequence, master, exp_avg,
                            exp_avg_sq, param16, step_counter, hp: zero_adam_hparams | dict,
                            loss_scale: float, clip: float, stream=None) -> None:
    """The shard step without a plan and without allocating anything (see zero.h): for
    callers that cannot allocate device memory when they step. ``step_counter`` is a
    one-element int64 device tensor (or address) holding the optimizer step counter."""
    if isinstance(hp, dict):
        hp = zero_adam_hparams(**hp)
    _check(_lib.zero_shard_step_noalloc(nd, n, n_valid, _ptrs(grads), _addr(master),
                                        _addr(exp_avg), _addr(exp_avg_sq), _addr(param16),
                                        _addr(step_counter), ctypes.byref(hp), loss_scale,
                                        clip, _stream(stream)))
