"""Python binding of libzero, the GB300 ZeRO shard-step library (include/zero.h).

Argument marshalling only: every step of the path runs in the library's CUDA kernels.
Functions carry the C names; they accept torch tensors (their ``data_ptr()`` is passed)
or raw integer addresses, and raise :class:`ZeroError` on a non-zero return code.
The first call loads ``libzero.so`` and raises if it has not been built
(``python -m sharded_emulated_reduce_gb300.build``); there is no fallback. The environment
variable ZERO_LIBZERO names another build of the library to load instead (the
bounds-checked ``libzero_checked.so`` in tests).
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("ZERO_LIBZERO") or os.path.join(_HERE, "libzero.so")

ZERO_OK = 0
ZERO_EINVAL = -1
ZERO_EALIGN = -2
ZERO_EUNBOUND = -3
ZERO_ECUDA = -4
ZERO_EDEVICE = -5
ZERO_MAX_ND = 256
ZERO_STATS_WORDS = 8
ZERO_PROF_KINDS = 5
ZERO_NOALLOC_MAX_SPAN = 4194304
PROF_REDUCE, PROF_UPDATE, PROF_FINALIZE, PROF_GATHER, PROF_STEP = range(5)


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
                ("loss_scale", ctypes.c_float)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_ if not k.startswith("reserved")}


class zero_loss_scaler(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("good_steps", ctypes.c_int32),
                ("growth_factor", ctypes.c_float), ("backoff_factor", ctypes.c_float),
                ("growth_interval", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_ if not k.startswith("reserved")}


class zero_plan_state(ctypes.Structure):
    _fields_ = [("step", ctypes.c_int64), ("scaler", zero_loss_scaler)]

    def as_dict(self) -> dict:
        return {"step": self.step, "scaler": self.scaler.as_dict()}


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
    "zero_gather_layers_events": ([_P, ctypes.POINTER(_I64), _I32, _PP, _PP, _PP, _P],
                                  ctypes.c_int),
    "zero_memory_bytes": ([_I64, _I32, _I32, _I32, ctypes.POINTER(_I64)], ctypes.c_int),
    "zero_gather_status": ([_P, ctypes.POINTER(_I32)], ctypes.c_int),
    "zero_profile_enable": ([_P, _I32], ctypes.c_int),
    "zero_profile_read": ([_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I64), _I32],
                          ctypes.c_int),
    "zero_shard_step_noalloc": ([_I32, _I64, _I64, _PP, _P, _P, _P, _P, _P,
                                 ctypes.POINTER(zero_adam_hparams), _F, _F, _P], ctypes.c_int),
    "zero_noalloc_step_result": ([_P, ctypes.POINTER(zero_step_info)], ctypes.c_int),
    "zero_plan_set_scaler": ([_P, ctypes.POINTER(zero_loss_scaler)], ctypes.c_int),
    "zero_loss_scale_ptr": ([_P, ctypes.POINTER(_P)], ctypes.c_int),
    "zero_plan_get_state": ([_P, ctypes.POINTER(zero_plan_state)], ctypes.c_int),
    "zero_plan_set_state": ([_P, ctypes.POINTER(zero_plan_state)], ctypes.c_int),
    "zero_selftest_wait": ([ctypes.c_uint32, ctypes.POINTER(_I32)], ctypes.c_int),
    "zero_selftest_grid_barrier": ([ctypes.c_uint32, _I32, ctypes.POINTER(_I32)], ctypes.c_int),
    "zero_bounds_check": ([_I32, ctypes.POINTER(_I32), ctypes.POINTER(_I32),
                           ctypes.POINTER(_I64)], ctypes.c_int),
    "zero_selftest_bounds": ([], ctypes.c_int),
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


def zero_gather_status(plan: Plan) -> int:
    """Wait for the plan's last gather; 0 if it finished (raises ZeroError otherwise)."""
    st = _I32()
    _check(_lib.zero_gather_status(plan, ctypes.byref(st)))
    return st.value


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
    least significant first, word 5 the count of reduce CTAs whose bounded wait expired
    (0 here), words 6..7 zero."""
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


def zero_noalloc_step_result(stream=None) -> zero_step_info:
    """Result of the last allocation-free step on the current device (waits for
    ``stream``); raises ZeroError with ZERO_EDEVICE if that step reported a failure."""
    info = zero_step_info()
    _check(_lib.zero_noalloc_step_result(_stream(stream), ctypes.byref(info)))
    return info


# ------------------------------------------------------------------------------------
# Dynamic loss scale and checkpoints

def zero_plan_set_scaler(plan: Plan, scale: float = 65536.0, growth_factor: float = 2.0,
                         backoff_factor: float = 0.5, growth_interval: int = 2000,
                         good_steps: int = 0) -> None:
    """Turn the device-resident loss scaler on (growth_interval >= 1) or off (0). While it
    is on, pass loss_scale = 0 to the step calls."""
    c = zero_loss_scaler(scale, good_steps, growth_factor, backoff_factor, growth_interval, 0)
    _check(_lib.zero_plan_set_scaler(plan, ctypes.byref(c)))


def zero_loss_scale_ptr(plan: Plan) -> int:
    """Device address of the current fp32 loss scale."""
    p = ctypes.c_void_p()
    _check(_lib.zero_loss_scale_ptr(plan, ctypes.byref(p)))
    return p.value


def zero_plan_get_state(plan: Plan) -> zero_plan_state:
    st = zero_plan_state()
    _check(_lib.zero_plan_get_state(plan, ctypes.byref(st)))
    return st


def zero_plan_set_state(plan: Plan, state: zero_plan_state) -> None:
    _check(_lib.zero_plan_set_state(plan, ctypes.byref(state)))


def zero_checkpoint_save(path: str, plan: Plan, master, exp_avg, exp_avg_sq, param16) -> None:
    """Write one span's checkpoint: the plan's state and the raw bytes of its four bound
    buffers (torch tensors on the device), as an uncompressed .npz file."""
    import numpy as np
    st = zero_plan_get_state(plan)
    arrays = {name: t.detach().contiguous().view(-1).view(torch_uint8()).cpu().numpy()
              for name, t in (("master", master), ("exp_avg", exp_avg),
                              ("exp_avg_sq", exp_avg_sq), ("param16", param16))}
    sc = st.scaler
    meta = np.array([st.step, sc.good_steps, sc.growth_interval], dtype=np.int64)
    fmeta = np.array([sc.scale, sc.growth_factor, sc.backoff_factor], dtype=np.float32)
    geom = np.array([plan.n_params, plan.nd, plan.stage, plan.align], dtype=np.int64)
    with open(path, "wb") as f:
        np.savez(f, meta=meta, fmeta=fmeta, geom=geom, **arrays)


def zero_checkpoint_load(path: str, plan: Plan, master, exp_avg, exp_avg_sq, param16) -> None:
    """Restore a checkpoint written by zero_checkpoint_save into the given device buffers
    (already bound to ``plan``, same sizes) and the plan's state."""
    import numpy as np
    import torch
    with np.load(path) as z_:
        geom = [int(x) for x in z_["geom"]]
        if geom != [plan.n_params, plan.nd, plan.stage, plan.align]:
            raise ZeroError(ZERO_EINVAL, f"checkpoint is for plan {geom}")
        for name, t in (("master", master), ("exp_avg", exp_avg), ("exp_avg_sq", exp_avg_sq),
                        ("param16", param16)):
            raw = torch.from_numpy(z_[name].copy())
            dst = t.view(-1).view(torch.uint8)
            if raw.numel() != dst.numel():
                raise ZeroError(ZERO_EINVAL, f"checkpoint {name} has {raw.numel()} bytes, "
                                             f"buffer has {dst.numel()}")
            dst.copy_(raw)
        meta, fmeta = z_["meta"], z_["fmeta"]
    torch.cuda.synchronize()
    st = zero_plan_state()
    st.step = int(meta[0])
    st.scaler = zero_loss_scaler(float(fmeta[0]), int(meta[1]), float(fmeta[1]), float(fmeta[2]),
                                 int(meta[2]), 0)
    zero_plan_set_state(plan, st)


def torch_uint8():
    import torch
    return torch.uint8


# ------------------------------------------------------------------------------------
# Layer-by-layer gather with completion events (ZeRO-3 prefetch)

def make_layer_events(n: int, timing: bool = False) -> list:
    """n torch.cuda.Event objects with their CUDA events already created (recorded once on
    the current stream), ready to be passed to zero_gather_layers_events."""
    import torch
    evs = [torch.cuda.Event(enable_timing=timing) for _ in range(n)]
    s = torch.cuda.current_stream()
    for ev in evs:
        ev.record(s)
    return evs


def _event_handle(ev) -> int:
    if ev is None:
        return 0
    if isinstance(ev, int):
        return ev
    h = int(ev.cuda_event)
    if not h:
        raise ZeroError(ZERO_EINVAL, "event has no CUDA event yet: record it once first "
                                     "(make_layer_events does)")
    return h


def zero_gather_layers_events(plan: Plan, layer_offsets: Sequence[int], shards: Sequence,
                              layer_dst: Sequence, events: Sequence, stream=None) -> None:
    """The gather layer by layer; events[l] (a torch.cuda.Event made by make_layer_events,
    a raw cudaEvent_t address, or None) is recorded when layer l has been copied."""
    n_layers = len(layer_offsets) - 1
    if len(events) != n_layers:
        raise ZeroError(ZERO_EINVAL, f"need {n_layers} events, got {len(events)}")
    offs = (_I64 * len(layer_offsets))(*[int(x) for x in layer_offsets])
    evs = (ctypes.c_void_p * n_layers)(*[_event_handle(e) for e in events])
    _check(_lib.zero_gather_layers_events(plan, offs, n_layers, _ptrs(shards),
                                          _ptrs(layer_dst), evs, _stream(stream)))


def zero_prefetch_layers(plan: Plan, layer_offsets: Sequence[int], shards: Sequence,
                         layer_dst: Sequence, stream=None, timing: bool = False) -> list:
    """Gather every layer with one C call and return one torch.cuda.Event per layer,
    recorded when that layer has been copied (with ``timing``, events that can be timed).
    A consumer stream that waits on event l can start on layer l while later layers are
    still being gathered: the "dynamic communication schedule" of the ZeRO method entry,
    in which the all-gather of the next layers runs ahead of the work on the current
    one."""
    events = make_layer_events(len(layer_offsets) - 1, timing=timing)
    zero_gather_layers_events(plan, layer_offsets, shards, layer_dst, events, stream)
    return events


def zero_selftest_wait(polls: int = 4096) -> int:
    """Run the bounded-wait self-test; 1 means the wait expired and was reported."""
    out = _I32()
    _check(_lib.zero_selftest_wait(polls, ctypes.byref(out)))
    return out.value


def zero_bounds_check(reset: bool = False) -> dict:
    """The bounds report of a bounds-checked build: {"enabled", "site", "offset"}; site 0
    means no access fell outside its buffer (always 0 in the normal build)."""
    en, site, off = _I32(), _I32(), _I64()
    _check(_lib.zero_bounds_check(1 if reset else 0, ctypes.byref(en), ctypes.byref(site),
                                  ctypes.byref(off)))
    return {"enabled": en.value, "site": site.value, "offset": off.value}


def zero_selftest_bounds() -> None:
    """Run the bounds self-test (see zero.h): a checked build then reports site 11."""
    _check(_lib.zero_selftest_bounds())


def zero_selftest_grid_barrier(polls: int = 4096, skip_one: bool = True) -> int:
    """Run the grid-barrier self-test: 0 means it was met with the right sums, 1 that it
    gave up and reported it, 2 that it was met with wrong sums."""
    out = _I32()
    _check(_lib.zero_selftest_grid_barrier(polls, 1 if skip_one else 0, ctypes.byref(out)))
    return out.value
