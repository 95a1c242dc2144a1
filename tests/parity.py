"""Parity harness: drive the GPU library and the CPU oracle on the same seeded inputs.

Expected values come only from the oracle, fed with the input bytes (gradients, initial
state) that the seeded generator wrote. Three modes:

* full: every element of every output is compared (sizes the oracle finishes in
  seconds);
* full_parallel: the same comparison of every element, with the oracle's step run over
  slices of the span on all host threads (bench.PartitionedOracle, bit-identical to one
  oracle step: the slices' integer statistics are added exactly before the scalars are
  taken), for full-size workloads whose inputs and state fit in host memory;
* sampled: the oracle streams all gradients through its reduce and exact sum of squares
  (the global norm and overflow flag need the whole span), then follows a sample of
  elements through every step with those scalars.

Bar: bit-exact overflow flag, skip decision, step counter and sum of squares; master,
exp_avg and exp_avg_sq within 1e-6 relative per element; param16 within 1 fp16 ulp;
global norm within 1e-5 relative. With the fixed operation order the step is also
expected to be bit-exact, and ``exact`` reports whether it was.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

import oracle
import sharded_emulated_reduce_gb300 as z
from synth import workloads as wl

THREADS = max(1, min(16, os.cpu_count() or 1))


def hyper(w: wl.Workload) -> oracle.Hyper:
    return oracle.Hyper(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
                        weight_decay=w.weight_decay)


def h16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_state_close(name, got, exp, idx=None):
    """master/m/v: 1e-6 relative per element (exact zeros must match exactly)."""
    got = np.asarray(got, dtype=np.float32)
    exp = np.asarray(exp, dtype=np.float32)
    both_nan = np.isnan(got) & np.isnan(exp)
    err = np.abs(got.astype(np.float64) - exp.astype(np.float64))
    tol = 1e-6 * np.abs(exp.astype(np.float64))
    bad = ~both_nan & ~(err <= tol)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        where = i if idx is None else int(idx[i])
        raise AssertionError(f"{name}: {int(bad.sum())} elements off; first at {where}: "
                             f"got {got[i]!r} expected {exp[i]!r}")


def f16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in representable fp16 steps (monotone integer mapping of the bits)."""
    def key(h):
        h = h.astype(np.int32)
        return np.where(h & 0x8000, 0x8000 - h, h)  # negative values mirrored below zero
    return np.abs(key(a) - key(b))


def assert_p16_close(got, exp, idx=None):
    d = f16_ulp_distance(np.asarray(got, np.uint16), np.asarray(exp, np.uint16))
    if (d > 1).any():
        i = int(np.flatnonzero(d > 1)[0])
        where = i if idx is None else int(idx[i])
        raise AssertionError(f"param16: {int((d > 1).sum())} elements beyond 1 ulp; first at "
                             f"{where}: got {got[i]:#06x} expected {exp[i]:#06x}")


def assert_info_matches(info: z.zero_step_info, sc: oracle.Scalars):
    assert info.overflow == sc.overflow, (info.overflow, sc.overflow)
    assert info.skipped == sc.skipped
    assert info.step == sc.step, (info.step, sc.step)
    assert info.status == 0
    if sc.overflow:
        assert np.isinf(info.global_norm)
        return
    assert info.sum_sq == sc.ss, (info.sum_sq, sc.ss)   # exact by construction
    assert info.global_norm == pytest_approx(sc.norm, 1e-5)
    assert np.float32(info.scale) == np.float32(sc.s)
    assert np.float32(info.bc1) == np.float32(sc.bc1)
    assert np.float32(info.bc2) == np.float32(sc.bc2)


def assert_state_full(name, got, exp, chunk=1 << 24) -> bool:
    """Every element of a full-size fp32 state array: True if bit-identical, else checked
    chunk by chunk at the 1e-6 relative bar (and False)."""
    if np.array_equal(got.view(np.uint32), exp.view(np.uint32)):
        return True
    for a in range(0, len(got), chunk):
        assert_state_close(name, got[a:a + chunk], exp[a:a + chunk],
                           np.arange(a, min(a + chunk, len(got))))
    return False


def assert_p16_full(got, exp, chunk=1 << 24) -> bool:
    if np.array_equal(got, exp):
        return True
    for a in range(0, len(got), chunk):
        assert_p16_close(got[a:a + chunk], exp[a:a + chunk], np.arange(a, min(a + chunk, len(got))))
    return False


def pytest_approx(x, rel):
    import pytest
    return pytest.approx(x, rel=rel)


# ------------------------------------------------------------------------------------
# streamed oracle statistics over device-resident gradients

def oracle_span_stats(grads: list[torch.Tensor], n_valid: int, chunk: int = 1 << 23) -> tuple[int, int]:
    """(non-finite count, exact sum of squares) of the rank-order sum over the first
    n_valid elements, computed by the oracle on chunks copied to the host."""
    starts = list(range(0, n_valid, chunk))

    def work(a):
        b = min(a + chunk, n_valid)
        host = [h16(g[a:b]) for g in grads]
        gsum = oracle.reduce(host)
        return oracle.stats(gsum)

    bad = 0
    ss = 0
    with ThreadPoolExecutor(THREADS) as ex:
        for b_, s_ in ex.map(work, starts):
            bad += b_
            ss += s_
    return bad, ss


@dataclass
class Sample:
    idx: np.ndarray           # span-relative element indices (real parameters only)
    master: np.ndarray
    m: np.ndarray
    v: np.ndarray
    p16: np.ndarray


def sample_indices(n_valid: int, s: int, count: int = 4096, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = set(rng.integers(0, n_valid, count).tolist())
    for i in [0, 1, 7, 8, 9, n_valid - 9, n_valid - 8, n_valid - 1]:
        if 0 <= i < n_valid:
            pick.add(i)
    k = 1
    while k * s <= n_valid:  # shard boundaries inside the span
        for d in (-1, 0):
            if 0 <= k * s + d < n_valid:
                pick.add(k * s + d)
        k += 1
    return np.array(sorted(pick), dtype=np.int64)


def device_words(addr: int, n: int) -> np.ndarray:
    """n int64 words at a raw device address, read with the CUDA runtime's cudaMemcpy."""
    import ctypes
    cudart = ctypes.CDLL("libcudart.so.13")
    out = np.zeros(n, dtype=np.int64)
    rc = cudart.cudaMemcpy(ctypes.c_void_p(out.ctypes.data), ctypes.c_void_p(addr),
                           ctypes.c_size_t(8 * n), 2)  # cudaMemcpyDeviceToHost
    assert rc == 0, rc
    return out


def take(t: torch.Tensor, idx: np.ndarray) -> torch.Tensor:
    return t[torch.as_tensor(idx, device=t.device)]


@dataclass
class Runner:
    """One workload on the device through the C ABI, followed by the oracle."""
    w: wl.Workload
    mode: str = "full"                      # or "full_parallel", "sampled"
    steps: int | None = None
    results: list = field(default_factory=list)
    exact: bool = True

    def run(self) -> "Runner":
        w = self.w
        steps = w.steps if self.steps is None else self.steps
        first, n_span, n_valid = w.span()
        _, s = w.layout()
        hp = hyper(w)
        master, m, v, p16, ws = wl.make_state(w)
        torch.cuda.synchronize()
        plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
        z.zero_plan_bind(plan, w.r0, w.r1, master, m, v, p16, ws, 0)
        if self.mode in ("full", "full_parallel"):
            om, omm, ov, op = f32(master).copy(), f32(m).copy(), f32(v).copy(), h16(p16).copy()
            if self.mode == "full_parallel":
                import bench
                par = bench.PartitionedOracle(n_valid, THREADS)
        else:
            idx = sample_indices(n_valid, s)
            smp = Sample(idx, f32(take(master, idx)).copy(), f32(take(m, idx)).copy(),
                         f32(take(v, idx)).copy(), h16(take(p16, idx)).copy())
        t = 0
        grads = [torch.empty(n_span, dtype=torch.float16, device="cuda") for _ in range(w.nd)]
        z.zero_profile_enable(plan, True)  # tells the one-launch steps from the others
        for step in range(steps):
            wl.fill_grads(w, step, grads)
            z.zero_shard_step(plan, w.r0, w.r1, grads, w.loss_scale, w.clip)
            info = z.zero_step_result(plan)
            one_launch = z.zero_profile_read(plan, reset=True)[1][z.PROF_STEP] > 0
            if self.mode == "full":
                host = [h16(g) for g in grads]
                sc = oracle.step(host, om, omm, ov, op, w.loss_scale, w.clip, hp, t,
                                 n_valid=n_valid)
                assert_info_matches(info, sc)
                if not sc.skipped and not one_launch:
                    # the two-kernel step leaves the rank-order sums in the workspace (the
                    # one-launch step keeps them on chip): compare them bit for bit
                    gs = oracle.reduce(host, n_valid)
                    assert np.array_equal(f32(ws)[:n_valid].view(np.uint32),
                                          gs[:n_valid].view(np.uint32))
                gm, gmm, gv, gp = f32(master), f32(m), f32(v), h16(p16)
                sl = slice(0, n_valid)
                assert_state_close("master", gm[sl], om[sl])
                assert_state_close("exp_avg", gmm[sl], omm[sl])
                assert_state_close("exp_avg_sq", gv[sl], ov[sl])
                assert_p16_close(gp[sl], op[sl])
                # padding starts at zero and is never touched by the library
                assert not gm[n_valid:].any() and not gmm[n_valid:].any()
                assert not gv[n_valid:].any() and not gp[n_valid:].any()
                self.exact &= (np.array_equal(gm.view(np.uint32), om.view(np.uint32)) and
                               np.array_equal(gmm.view(np.uint32), omm.view(np.uint32)) and
                               np.array_equal(gv.view(np.uint32), ov.view(np.uint32)) and
                               np.array_equal(gp, op))
            elif self.mode == "full_parallel":
                nv = n_valid
                host = [h16(g)[:nv] for g in grads]
                sc = par.step(host, om[:nv], omm[:nv], ov[:nv], op[:nv], w.loss_scale, w.clip,
                              hp, t, keep_sums=True)
                del host
                assert_info_matches(info, sc)
                if not sc.skipped and not one_launch:
                    gws = f32(ws)
                    for sl, gs in zip(par.slices, par.sums):
                        assert np.array_equal(gws[sl].view(np.uint32), gs.view(np.uint32))
                    del gws
                for name, got, exp in (("master", master, om), ("exp_avg", m, omm),
                                       ("exp_avg_sq", v, ov)):
                    g_ = f32(got)
                    self.exact &= assert_state_full(name, g_[:nv], exp[:nv])
                    assert not g_[nv:].any()  # padding is never touched
                    del g_
                gp = h16(p16)
                self.exact &= assert_p16_full(gp[:nv], op[:nv])
                assert not gp[nv:].any()
                del gp
            else:
                bad, ss = oracle_span_stats(grads, n_valid)
                sc = oracle.scalars(bad, ss, w.loss_scale, w.clip, hp, t)
                assert_info_matches(info, sc)
                idx = smp.idx
                host = [h16(take(g, idx)) for g in grads]
                gs = oracle.reduce(host)
                if not sc.skipped:
                    assert np.array_equal(f32(take(ws, idx)).view(np.uint32), gs.view(np.uint32))
                oracle.adam(gs, smp.master, smp.m, smp.v, smp.p16, sc)
                gm, gmm, gv, gp = (f32(take(master, idx)), f32(take(m, idx)), f32(take(v, idx)),
                                   h16(take(p16, idx)))
                assert_state_close("master", gm, smp.master, idx)
                assert_state_close("exp_avg", gmm, smp.m, idx)
                assert_state_close("exp_avg_sq", gv, smp.v, idx)
                assert_p16_close(gp, smp.p16, idx)
                self.exact &= (np.array_equal(gm.view(np.uint32), smp.master.view(np.uint32)) and
                               np.array_equal(gp, smp.p16))
            t = sc.step
            self.results.append(info.as_dict())
        if self.mode == "full_parallel":
            par.close()
        self.state = (master, m, v, p16, ws)
        self.plan = plan
        return self
