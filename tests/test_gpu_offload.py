"""GPU: optimizer state in Grace host memory (ZeRO-Offload/Infinity lineage, named on the
ZeRO pages: "Legacy", CPU/NVMe offload). On a GB300 the kernels address pinned host
memory directly over NVLink-C2C, so the same step and gather run with the master weights,
moments and fp16 parameters (or the fp16 shards) in host memory; results must be the
same bits as with device-resident state."""
import numpy as np
import pytest
import torch

import oracle
import sharded_emulated_reduce_gb300 as z
from synth import workloads as wl

from parity import assert_info_matches, f32, h16, hyper

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [1_000_003, 6_000_001])
def test_step_with_state_in_pinned_host_memory(n):
    # 1,000,003 parameters run the one-launch step; 6,000,001 (above its limit on a
    # 152-SM part) run the reduce and the bulk-copy update kernel, whose TMA loads and
    # stores then address pinned host memory. The second step carries a +inf in rank 3
    # and must leave the host-resident state untouched.
    w = wl.Workload("offload", cfg=500, n=n, nd=8, align=8, stage=2, r0=0, r1=8,
                    loss_scale=65536.0, grad_sigma=1e-3, clip=1.0, steps=3, m_sigma=1e-3,
                    v_sigma=1e-6, inject=((1, 3, wl.POS_INF, n // 3),))
    first, n_span, n_valid = w.span()
    dev_state = wl.make_state(w)
    host_state = [t.cpu().pin_memory() for t in dev_state[:4]]
    om, omm, ov, op = (f32(dev_state[0]).copy(), f32(dev_state[1]).copy(),
                       f32(dev_state[2]).copy(), h16(dev_state[3]).copy())
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, 0, w.nd, *host_state, dev_state[4], 0)  # workspace stays in HBM
    z.zero_profile_enable(plan, True)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    one_launch = n_span // 8 <= 3072 * sms
    t = 0
    for step in range(w.steps):
        grads = wl.make_grads(w, step)
        z.zero_shard_step(plan, 0, w.nd, grads, w.loss_scale, w.clip)
        info = z.zero_step_result(plan)
        sc = oracle.step([h16(g) for g in grads], om, omm, ov, op, w.loss_scale, w.clip,
                         hyper(w), t, n_valid=n_valid)
        assert_info_matches(info, sc)
        assert sc.skipped == (step == 1)
        t = sc.step
        torch.cuda.synchronize()
        assert np.array_equal(host_state[0].numpy().view(np.uint32), om.view(np.uint32))
        assert np.array_equal(host_state[1].numpy().view(np.uint32), omm.view(np.uint32))
        assert np.array_equal(host_state[2].numpy().view(np.uint32), ov.view(np.uint32))
        assert np.array_equal(host_state[3].view(torch.int16).numpy().view(np.uint16), op)
    launches = z.zero_profile_read(plan)[1]
    if one_launch:
        assert launches[z.PROF_STEP] == w.steps and launches[z.PROF_UPDATE] == 0
    else:
        assert launches[z.PROF_UPDATE] == w.steps and launches[z.PROF_STEP] == 0
    plan.close()


def test_gather_from_shards_in_pinned_host_memory():
    n, nd = 640_000, 8
    _, s = oracle.partition(n, nd, 8)
    shards = [torch.randint(-30000, 30000, (s,), dtype=torch.int16).pin_memory() for _ in range(nd)]
    offs = [0, 100_003, 400_000, n]
    dst = [torch.empty(offs[l + 1] - offs[l], dtype=torch.int16, device="cuda") for l in range(3)]
    plan = z.zero_plan_create(n, nd, 3, 8, dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                                weight_decay=0.0))
    z.zero_gather_layers(plan, offs, shards, dst)
    torch.cuda.synchronize()
    exp = oracle.gather([x.numpy().view(np.uint16) for x in shards], s, offs)
    for d, e in zip(dst, exp):
        assert np.array_equal(h16(d), e)
    plan.close()


@pytest.mark.parametrize("nd", [4, 8, 64])
def test_step_reads_gradients_from_pinned_host_memory(nd):
    # the end-to-end bench's zero-copy mode: the gradient contributions stay in pinned
    # Grace memory and the reduce reads them over NVLink-C2C (register loads for 4 ranks,
    # TMA bulk loads for 8 and 64); the span is above the one-launch limit, so the reduce
    # and update kernels run, and every element must match the oracle
    n = 4_500_007 if nd <= 8 else 4_000_037
    w = wl.Workload("hostgrads", cfg=520 + nd, n=n, nd=nd, align=8, stage=2, r0=0, r1=nd,
                    loss_scale=1024.0, grad_sigma=1e-3, clip=1.0, steps=2, m_sigma=1e-3,
                    v_sigma=1e-6)
    first, n_span, n_valid = w.span()
    master, m, v, p16, ws = wl.make_state(w)
    om, omm, ov, op = f32(master).copy(), f32(m).copy(), f32(v).copy(), h16(p16).copy()
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, 0, w.nd, master, m, v, p16, ws, 0)
    z.zero_profile_enable(plan, True)
    t = 0
    for step in range(w.steps):
        host = [g.cpu().pin_memory() for g in wl.make_grads(w, step)]
        z.zero_shard_step(plan, 0, w.nd, host, w.loss_scale, w.clip)
        info = z.zero_step_result(plan)
        sc = oracle.step([g.view(torch.int16).numpy().view(np.uint16) for g in host], om, omm,
                         ov, op, w.loss_scale, w.clip, hyper(w), t, n_valid=n_valid)
        assert_info_matches(info, sc)
        t = sc.step
    assert z.zero_profile_read(plan)[1][z.PROF_REDUCE] == w.steps  # the two-kernel path
    assert np.array_equal(f32(master).view(np.uint32), om.view(np.uint32))
    assert np.array_equal(f32(m).view(np.uint32), omm.view(np.uint32))
    assert np.array_equal(f32(v).view(np.uint32), ov.view(np.uint32))
    assert np.array_equal(h16(p16), op)
    plan.close()
