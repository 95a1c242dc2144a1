"""GPU: the device-resident dynamic loss scaler against the oracle's rule, and bit-exact
checkpoint/resume of a span (the plan's step counter and scaler plus its four buffers)."""
import os
import tempfile

import numpy as np
import pytest
import torch

import oracle
import sharded_emulated_reduce_gb300 as z
from synth import GRAD, fill
from synth import workloads as wl

from parity import assert_info_matches, f32, h16, hyper

pytestmark = pytest.mark.gpu


def workload(**kw):
    base = dict(name="state", cfg=400, n=200_003, nd=4, align=8, stage=2, r0=0, r1=4,
                loss_scale=0.0, grad_sigma=1e-3, clip=1.0, steps=8, m_sigma=1e-3, v_sigma=1e-6)
    base.update(kw)
    return wl.Workload(**base)


def grads_at_scale(w, step, scale, out, inject=None):
    first, n_span, _ = w.span()
    for k, t in enumerate(out):
        fill(t, wl.key(w, GRAD, step, k), w.grad_sigma * scale, start=first, n_valid=w.n)
    if inject is not None and step in inject:
        out[inject[step]].view(torch.int16)[777] = 0x7C00


def test_dynamic_scaler_follows_the_oracle_rule():
    w = workload()
    first, n_span, n_valid = w.span()
    master, m, v, p16, ws = wl.make_state(w)
    om, omm, ov, op = f32(master).copy(), f32(m).copy(), f32(v).copy(), h16(p16).copy()
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, 0, w.nd, master, m, v, p16, ws, 0)
    z.zero_plan_set_scaler(plan, scale=65536.0, growth_factor=2.0, backoff_factor=0.5,
                           growth_interval=2)
    with pytest.raises(z.ZeroError):
        z.zero_shard_step(plan, 0, w.nd, [ws] * w.nd, 1024.0, 1.0)  # must pass loss_scale 0
    scale, good, t = 65536.0, 0, 0
    inject = {2: 1, 5: 3}
    grads = [torch.empty(n_span, dtype=torch.float16, device="cuda") for _ in range(w.nd)]
    for step in range(w.steps):
        dev_scale = z.zero_plan_get_state(plan).scaler.scale
        assert dev_scale == np.float32(scale)
        grads_at_scale(w, step, scale, grads, inject)
        z.zero_shard_step(plan, 0, w.nd, grads, 0.0, w.clip)
        info = z.zero_step_result(plan)
        assert info.loss_scale == np.float32(scale)
        sc = oracle.step([h16(g) for g in grads], om, omm, ov, op, scale, w.clip, hyper(w), t,
                         n_valid=n_valid)
        assert_info_matches(info, sc)
        t = sc.step
        scale, good = oracle.scaler_update(scale, good, bool(sc.overflow), 2.0, 0.5, 2)
        st = z.zero_plan_get_state(plan)
        assert (st.step, st.scaler.scale, st.scaler.good_steps) == (t, np.float32(scale), good)
    assert np.array_equal(f32(master).view(np.uint32), om.view(np.uint32))
    assert np.array_equal(h16(p16), op)
    # the scale's device address holds the same value
    addr = z.zero_loss_scale_ptr(plan)
    import ctypes
    val = ctypes.c_float()
    cudart = ctypes.CDLL("libcudart.so.13")
    assert cudart.cudaMemcpy(ctypes.byref(val), ctypes.c_void_p(addr), ctypes.c_size_t(4), 2) == 0
    assert val.value == np.float32(scale)
    plan.close()


def run_steps(w, plan, state, steps, scale_of_step):
    first, n_span, _ = w.span()
    grads = [torch.empty(n_span, dtype=torch.float16, device="cuda") for _ in range(w.nd)]
    infos = []
    for step in steps:
        sc = z.zero_plan_get_state(plan).scaler.scale
        grads_at_scale(w, step, sc, grads, {2: 0})
        z.zero_shard_step(plan, 0, w.nd, grads, 0.0, w.clip)
        infos.append(z.zero_step_result(plan).as_dict())
    return infos


def test_checkpoint_resume_is_bit_exact():
    w = workload(cfg=410)
    straight = wl.make_state(w)
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, 0, w.nd, *straight, 0)
    z.zero_plan_set_scaler(plan, scale=4096.0, growth_interval=2)
    infos_a = run_steps(w, plan, straight, range(6), None)
    plan.close()

    first_half = wl.make_state(w)
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, 0, w.nd, *first_half, 0)
    z.zero_plan_set_scaler(plan, scale=4096.0, growth_interval=2)
    infos_b = run_steps(w, plan, first_half, range(3), None)
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "span0.npz")
        z.zero_checkpoint_save(path, plan, *first_half[:4])
        plan.close()
        del first_half
        resumed = [torch.full_like(t, 7) for t in wl.make_state(w)]
        plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
        z.zero_plan_bind(plan, 0, w.nd, *resumed, 0)
        z.zero_checkpoint_load(path, plan, *resumed[:4])
    infos_b += run_steps(w, plan, resumed, range(3, 6), None)
    assert infos_a == infos_b
    assert [x["skipped"] for x in infos_a] == [0, 0, 1, 0, 0, 0]
    for a, b in zip(straight[:4], resumed[:4]):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert z.zero_plan_get_state(plan).step == 5
    plan.close()
