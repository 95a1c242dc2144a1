"""The shard step that allocates nothing, checked against the plan-based step.

Some callers cannot allocate device memory at the moment they run the optimizer step:
their framework reserved all of HBM for its own pool at start-up, they run inside an
allocator hook, or they cannot afford the device-wide synchronisation cudaMalloc and
cudaFree may cause. zero_shard_step_noalloc serves them from a fixed scratch array
inside the library. Here two calls in a row must leave the same state and step counter
as zero_shard_step on identical inputs, within the tolerances of the other parity tests
(1e-6 relative for master/m/v, one fp16 ulp for the parameters), the companion
zero_noalloc_step_result must report the step (no device failure, the same norm and
counter), and a span longer than the array must be refused with a clear error. The test
stands alone: it needs nothing from the tests collected before it.
"""
import numpy as np
import pytest
import torch

import sharded_emulated_reduce_gb300 as z
from synth import workloads as wl

from parity import assert_p16_close, assert_state_close, f32, h16

pytestmark = pytest.mark.gpu


def one_launch_limit() -> int:
    """Largest span the one-launch step takes on this device: 3072 groups of 8 per SM."""
    return 8 * 3072 * torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("path", ["one_launch", "two_kernels"])
def test_noalloc_step_matches_plan_step_on_two_calls(path):
    # a span just below the one-launch limit, and the largest span the array holds, which
    # runs the reduce and update kernels whenever it is above that limit (it is on a
    # 152-SM GB300); the plan's launch counters show which path the equal-sized plan step
    # took, and the allocation-free step decides by the same rule
    limit = one_launch_limit()
    if path == "one_launch":
        n = min(limit, z.ZERO_NOALLOC_MAX_SPAN) - 7
    else:
        n = z.ZERO_NOALLOC_MAX_SPAN
        if n <= limit:
            pytest.skip("this device takes every span the array holds in one launch")
    w = wl.Workload("noalloc", cfg=300, n=n, nd=8, align=8, stage=2, r0=0, r1=8,
                    loss_scale=65536.0, grad_sigma=1e-3, clip=1.0, steps=2, m_sigma=1e-3,
                    v_sigma=1e-6)
    first, n_span, n_valid = w.span()
    assert n_span <= z.ZERO_NOALLOC_MAX_SPAN
    ref = wl.make_state(w)
    mine = [t.clone() for t in ref[:4]]
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, 0, w.nd, *ref, 0)
    z.zero_profile_enable(plan, True)
    counter = torch.zeros(1, dtype=torch.int64, device="cuda")
    grads = [torch.empty(n_span, dtype=torch.float16, device="cuda") for _ in range(w.nd)]
    for step in range(2):
        wl.fill_grads(w, step, grads)
        z.zero_shard_step(plan, 0, w.nd, grads, w.loss_scale, w.clip)
        info = z.zero_step_result(plan)
        z.zero_shard_step_noalloc(w.nd, n_span, n_valid, grads, *mine, counter, w.hparams(),
                                  w.loss_scale, w.clip)
        mine_info = z.zero_noalloc_step_result()
        assert info.skipped == 0 and mine_info.status == 0 and mine_info.skipped == 0
        assert int(counter.item()) == info.step == mine_info.step == step + 1
        assert mine_info.sum_sq == info.sum_sq and mine_info.global_norm == info.global_norm
        assert mine_info.clip_coef == info.clip_coef and mine_info.scale == info.scale
        for name, a, b in zip(("master", "exp_avg", "exp_avg_sq"), mine[:3], ref[:3]):
            assert_state_close(name, f32(a)[:n_valid], f32(b)[:n_valid])
            assert np.array_equal(f32(a).view(np.uint32), f32(b).view(np.uint32))
        assert_p16_close(h16(mine[3])[:n_valid], h16(ref[3])[:n_valid])
        assert np.array_equal(h16(mine[3]), h16(ref[3]))
    launches = z.zero_profile_read(plan)[1]
    if path == "one_launch":
        assert launches[z.PROF_STEP] == 2 and launches[z.PROF_UPDATE] == 0
    else:
        assert launches[z.PROF_UPDATE] == 2 and launches[z.PROF_STEP] == 0
    plan.close()


def test_noalloc_skips_an_overflow_step_and_keeps_the_counter():
    n, nd = 4096, 4
    master = torch.zeros(n, device="cuda")
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    p16 = torch.zeros(n, dtype=torch.float16, device="cuda")
    counter = torch.full((1,), 7, dtype=torch.int64, device="cuda")
    grads = [torch.ones(n, dtype=torch.float16, device="cuda") for _ in range(nd)]
    grads[2][100] = float("inf")
    z.zero_shard_step_noalloc(nd, n, n, grads, master, m, v, p16, counter,
                              dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0),
                              1.0, 0.0)
    info = z.zero_noalloc_step_result()
    assert info.overflow == 1 and info.skipped == 1 and info.status == 0 and info.step == 7
    assert int(counter.item()) == 7
    assert not master.any() and not m.any() and not v.any()


def test_noalloc_alternating_hyperparameters_follow_the_oracle():
    """Two optimizers with different hyperparameters step in turn through the one scratch
    array; the step-counter-only scalars it keeps between calls belong to one of them at
    a time, and each step must still match the oracle bit for bit."""
    import oracle
    n, nd = 8200, 4
    gen = torch.Generator().manual_seed(11)
    users = []
    for hp in (dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
               dict(lr=3e-4, beta1=0.5, beta2=0.95, eps=1e-6, weight_decay=0.0)):
        master = (torch.randn(n, generator=gen) * 0.02).float()
        users.append({"hp": hp, "master": master.cuda(), "m": torch.zeros(n, device="cuda"),
                      "v": torch.zeros(n, device="cuda"),
                      "p16": master.half().cuda(),
                      "counter": torch.zeros(1, dtype=torch.int64, device="cuda"),
                      "ref": [master.numpy().copy(), np.zeros(n, np.float32),
                              np.zeros(n, np.float32),
                              master.half().numpy().view(np.uint16).copy()],
                      "t": 0})
    for rnd in range(3):
        for u in users:
            g = [(torch.randn(n, generator=gen) * 1e-3 * 1024).half() for _ in range(nd)]
            z.zero_shard_step_noalloc(nd, n, n, [x.cuda() for x in g], u["master"], u["m"],
                                      u["v"], u["p16"], u["counter"], u["hp"], 1024.0, 0.1)
            sc = oracle.step([x.numpy().view(np.uint16) for x in g], *u["ref"], 1024.0, 0.1,
                             oracle.Hyper(**u["hp"]), u["t"])
            u["t"] = sc.step
            torch.cuda.synchronize()
            assert int(u["counter"].item()) == sc.step == rnd + 1
            for a, b in zip((u["master"], u["m"], u["v"]), u["ref"][:3]):
                assert np.array_equal(f32(a).view(np.uint32), b.view(np.uint32)), rnd
            assert np.array_equal(h16(u["p16"]), u["ref"][3]), rnd


def test_noalloc_refuses_spans_beyond_its_array():
    fake = [0x10000 + 0x1000 * k for k in range(4)]
    n = z.ZERO_NOALLOC_MAX_SPAN + 8
    with pytest.raises(z.ZeroError) as ei:
        z.zero_shard_step_noalloc(4, n, n, fake, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000,
                                  dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                       weight_decay=0.0), 1.0, 0.0)
    assert ei.value.code == z.ZERO_EINVAL
    assert "ZERO_NOALLOC_MAX_SPAN" in str(ei.value)
