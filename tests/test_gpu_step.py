"""GPU parity of the shard step through the C ABI against the oracle, element by element.

Sizes here are ones the oracle finishes in seconds: they span many CTAs and grid-stride
rounds, ragged shard tails (padding) and every rank count the kernels specialise.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import sharded_emulated_reduce_gb300 as z
from synth import workloads as wl

from parity import Runner, assert_info_matches, device_words, h16, f32, hyper

pytestmark = pytest.mark.gpu

TINY = wl.WORKLOADS["zero2_tiny_1m_nd4"]


def small(**kw) -> wl.Workload:
    base = dict(name="small", cfg=100, n=4099, nd=4, align=8, stage=2, r0=0, r1=4,
                loss_scale=1024.0, grad_sigma=1e-3, clip=1.0, steps=3, m_sigma=1e-3,
                v_sigma=1e-6)
    base.update(kw)
    return wl.Workload(**base)


def test_tiny_zero2_workload_all_steps_bit_exact():
    r = Runner(TINY).run()
    assert len(r.results) == TINY.steps and all(x["skipped"] == 0 for x in r.results)
    assert r.exact


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1023, 4099, 70001])
@pytest.mark.parametrize("nd", [1, 2, 3, 4, 5, 8, 16, 17, 32, 64, 100, 256])
def test_odd_shapes_and_rank_counts(n, nd):
    if n * nd > 2_000_000:
        n = 2_000_000 // nd
    r = Runner(small(n=n, nd=nd, r1=nd, cfg=101 + nd)).run()
    assert r.exact


@pytest.mark.parametrize("nd", [1, 2, 3, 4, 5, 7, 8, 9, 16, 24, 32, 33, 63, 64, 65, 128])
def test_two_kernel_path_every_reduce_variant(nd):
    # spans above the one-launch limit (3072 groups of 8 per SM): every branch of the
    # reduce's dispatch, the register-load reduce for fewer than 8 ranks (counts fixed at
    # compile time or read at run time) and the bulk-load reduce from 8 ranks on (fixed
    # counts 8, 16, 32, 64 and run-time counts up to 64 and beyond), then the update, over
    # two steps with a ragged tail
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = 8 * 3072 * sms + 37  # just past the one-launch limit, not a multiple of 8
    r = Runner(small(n=n, nd=nd, r1=nd, cfg=700 + nd), mode="full_parallel").run()
    assert r.exact


@pytest.mark.parametrize("align", [8, 16, 128])
@pytest.mark.parametrize("r0,r1", [(0, 1), (1, 3), (2, 3), (0, 3)])
def test_rank_subranges_and_alignment(align, r0, r1):
    w = small(n=10_000, nd=3, align=align, r0=r0, r1=r1, cfg=130 + align + r0 * 7 + r1)
    assert Runner(w).run().exact


def test_span_entirely_in_padding():
    # N = 5, Nd = 4, align = 8: shards 1..3 hold only padding
    w = small(n=5, nd=4, r0=2, r1=4, cfg=140)
    r = Runner(w).run()
    assert all(x["global_norm"] == 0.0 and x["step"] == i + 1 for i, x in enumerate(r.results))


@pytest.mark.parametrize("where", ["first", "middle", "last", "padding"])
@pytest.mark.parametrize("rank", ["first", "last"])
@pytest.mark.parametrize("value", [wl.POS_INF, wl.NEG_INF, wl.QNAN])
def test_overflow_injection(where, rank, value):
    n, nd = 4990, 5  # padded to 5000: ten padding elements
    idx = {"first": 0, "middle": n // 2, "last": n - 1, "padding": n + 3}[where]
    rk = 0 if rank == "first" else nd - 1
    w = small(n=n, nd=nd, r1=nd, steps=3, cfg=150, inject=((1, rk, value, idx),))
    r = Runner(w).run()
    skipped = [x["skipped"] for x in r.results]
    assert skipped == ([0, 0, 0] if where == "padding" else [0, 1, 0])
    assert [x["step"] for x in r.results] == ([1, 2, 3] if where == "padding" else [1, 1, 2])
    assert r.exact


@pytest.mark.parametrize("where", ["first", "last"])
@pytest.mark.parametrize("ls", [1024.0, 3.0])
def test_clip_off_overflow_and_applied_steps_in_one_launch(where, ls):
    # clipping off (the update's scale is then 1 / loss scale and needs no norm) in the
    # one-launch step: the overflow at step 1 must leave every state bit as it was, and
    # the applied steps must match the oracle
    n = 1_000_003
    idx = 0 if where == "first" else n - 1
    w = small(n=n, clip=0.0, loss_scale=ls, steps=3, cfg=157,
              inject=((1, 3, wl.POS_INF, idx),))
    r = Runner(w).run()
    assert [x["skipped"] for x in r.results] == [0, 1, 0]
    assert [x["step"] for x in r.results] == [1, 1, 2]
    assert all(x["clip_coef"] == 1.0 for x in r.results)
    assert r.exact


@pytest.mark.parametrize("path", ["one launch", "two kernels"])
def test_many_steps_stay_bit_exact(path):
    # hundreds of consecutive steps (the launch counts and scalar slots cycling, the bias
    # corrections at large t), two of them skipped by injected overflows: every element
    # of every output equals the oracle's, bit for bit, at every step
    if path == "one launch":
        w = dataclasses.replace(TINY, name="tiny_long", steps=1000,
                                inject=((57, 1, wl.POS_INF, 123), (211, 3, wl.QNAN, 777_777)))
    else:
        w = small(n=5_000_003, steps=200, cfg=158,
                  inject=((17, 0, wl.NEG_INF, 4_999_999), (64, 2, wl.POS_INF, 2_500_000)))
    r = Runner(w, mode="full_parallel").run()
    assert sum(x["skipped"] for x in r.results) == 2
    assert r.results[-1]["step"] == w.steps - 2
    assert r.exact


def test_opposite_infinities_in_two_ranks_make_nan_and_skip():
    w = small(n=3000, nd=4, steps=2, cfg=160,
              inject=((0, 0, wl.POS_INF, 1234), (0, 3, wl.NEG_INF, 1234)))
    r = Runner(w).run()
    assert [x["skipped"] for x in r.results] == [1, 0]


def test_clip_off_and_on_and_mean_loss_scale():
    for clip, ls in [(0.0, 1024.0), (1e-3, 1024.0), (1e6, 4096.0), (1.0, 4.0 * 1024.0)]:
        assert Runner(small(n=20_000, clip=clip, loss_scale=ls, cfg=170)).run().exact


@pytest.mark.parametrize("ls", [1000.0, 3.0, 98304.0, 0.7, 2.0 ** -20, 2.0 ** 40])
@pytest.mark.parametrize("n", [20_000, 5_000_003])
def test_loss_scales_powers_of_two_and_others(ls, n):
    # the norm and the unscale factor divide by the loss scale; a power of two is divided
    # by multiplying with its exact reciprocal, any other scale by a division: both must
    # give the oracle's bits (the fp16 gradients have sigma 1 whatever the scale); the
    # 5M span runs the reduce and update kernels, the 20K span the one-launch step
    w = small(n=n, loss_scale=ls, grad_sigma=1.0 / ls, clip=1.0, cfg=175)
    assert Runner(w).run().exact


def test_two_runs_are_bit_identical():
    outs = []
    for _ in range(2):
        r = Runner(small(n=300_000, nd=8, r1=8, cfg=180, steps=2)).run()
        outs.append([f32(t).copy() if t.dtype == torch.float32 else h16(t).copy()
                     for t in r.state[:4]])
        r.plan.close()
    for a, b in zip(*outs):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_split_reduce_update_equals_fused_step():
    w = small(n=200_000, nd=8, r1=8, cfg=190, steps=3)
    first, n_span, n_valid = w.span()
    states = []
    infos = []
    for split in (False, True):
        master, m, v, p16, ws = wl.make_state(w)
        plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
        z.zero_plan_bind(plan, w.r0, w.r1, master, m, v, p16, ws, 0)
        grads = [torch.empty(n_span, dtype=torch.float16, device="cuda") for _ in range(w.nd)]
        inf = []
        for step in range(w.steps):
            wl.fill_grads(w, step, grads)
            if split:
                z.zero_shard_reduce(plan, w.r0, w.r1, grads)
                words = z.zero_shard_stats(plan)
                assert words % 8 == 0
                z.zero_shard_update(plan, w.r0, w.r1, w.loss_scale, w.clip)
            else:
                z.zero_shard_step(plan, w.r0, w.r1, grads, w.loss_scale, w.clip)
            inf.append(z.zero_step_result(plan).as_dict())
        states.append([f32(master), f32(m), f32(v), h16(p16)])
        infos.append(inf)
        plan.close()
    assert infos[0] == infos[1]
    for a, b in zip(*states):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_exchange_buffer_holds_the_oracle_statistics():
    w = small(n=50_000, nd=4, cfg=200, steps=1)
    first, n_span, n_valid = w.span()
    master, m, v, p16, ws = wl.make_state(w)
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, 0, 4, master, m, v, p16, ws, 0)
    grads = wl.make_grads(w, 0)
    z.zero_shard_reduce(plan, 0, 4, grads)
    torch.cuda.synchronize()
    got = device_words(z.zero_shard_stats(plan), z.ZERO_STATS_WORDS).tolist()
    bad, ss = oracle.stats(oracle.reduce([h16(g) for g in grads], n_valid))
    assert got[0] == bad
    assert sum(got[1 + i] << (32 * i) for i in range(4)) == ss
    assert got[5:] == [0, 0, 0]


def test_profile_counts_every_launch():
    w = small(n=100_000, nd=4, cfg=210, steps=1)
    first, n_span, n_valid = w.span()
    master, m, v, p16, ws = wl.make_state(w)
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, 0, 4, master, m, v, p16, ws, 0)
    z.zero_profile_enable(plan, True)
    grads = wl.make_grads(w, 0)
    for _ in range(5):
        z.zero_shard_step(plan, 0, 4, grads, w.loss_scale, w.clip)
    z.zero_shard_reduce(plan, 0, 4, grads)
    z.zero_shard_update(plan, 0, 4, w.loss_scale, w.clip)
    ms, n = z.zero_profile_read(plan, reset=True)
    # 100,000 parameters fit the one-launch step (kind 4); the split call runs the reduce,
    # the finalize and the update
    assert n == [1, 1, 1, 0, 5] and all(ms[k] > 0 for k in (0, 1, 2, 4))
    ms, n = z.zero_profile_read(plan)
    assert n == [0] * z.ZERO_PROF_KINDS
    plan.close()


def test_profile_counts_the_next_step_scalars_of_a_full_wave_span():
    # a span that fills the reduce's wave computes the next step's scalars in a one-thread
    # kernel on the plan's second stream: one more launch of kind 2 per step
    w = small(n=5_000_000, nd=4, cfg=211, steps=1)
    master, m, v, p16, ws = wl.make_state(w)
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, 0, 4, master, m, v, p16, ws, 0)
    z.zero_profile_enable(plan, True)
    grads = wl.make_grads(w, 0)
    for _ in range(3):
        z.zero_shard_step(plan, 0, 4, grads, w.loss_scale, w.clip)
    ms, n = z.zero_profile_read(plan, reset=True)
    assert n[:3] == [3, 3, 3]
    plan.close()


def test_step_counter_continues_from_initial_step():
    w = small(n=4096, cfg=220, steps=1)
    first, n_span, n_valid = w.span()
    master, m, v, p16, ws = wl.make_state(w)
    om, omm, ov, op = f32(master).copy(), f32(m).copy(), f32(v).copy(), h16(p16).copy()
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, 0, 4, master, m, v, p16, ws, 41)
    grads = wl.make_grads(w, 0)
    z.zero_shard_step(plan, 0, 4, grads, w.loss_scale, w.clip)
    info = z.zero_step_result(plan)
    sc = oracle.step([h16(g) for g in grads], om, omm, ov, op, w.loss_scale, w.clip, hyper(w),
                     41, n_valid=n_valid)
    assert info.step == 42
    assert_info_matches(info, sc)
    assert np.array_equal(f32(master).view(np.uint32), om.view(np.uint32))


def test_wrong_device_state_and_stream_usage():
    w = small(n=4096, cfg=230, steps=1)
    master, m, v, p16, ws = wl.make_state(w)
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, 0, 4, master, m, v, p16, ws, 0)
    grads = wl.make_grads(w, 0)
    with pytest.raises(z.ZeroError) as ei:
        z.zero_shard_step(plan, 0, 3, grads, 1.0, 0.0)   # not the bound span
    assert ei.value.code == z.ZERO_EUNBOUND
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        z.zero_shard_step(plan, 0, 4, grads, w.loss_scale, w.clip)
    assert z.zero_step_result(plan).step == 1


def test_device_generator_matches_cpu_generator():
    import synth
    key = synth.stream_key(0, synth.GRAD, 7, 3, 2)
    for dtype, sigma in [(torch.float16, 65.536), (torch.float32, 0.02), (torch.float32, -1e-6)]:
        t = torch.empty(100_003, dtype=dtype, device="cuda")
        synth.fill(t, key, sigma, start=12345, n_valid=12345 + 90_000)
        if dtype == torch.float16:
            ref = synth.values_f16(key, sigma, 12345, 100_003, n_valid=12345 + 90_000)
            assert np.array_equal(h16(t), ref)
        else:
            ref = synth.values_f32(key, abs(sigma), 12345, 100_003, n_valid=12345 + 90_000,
                                   absolute=sigma < 0)
            assert np.array_equal(f32(t).view(np.uint32), ref.view(np.uint32))


def test_dist_step_in_one_process_group_equals_step():
    import os
    import socket
    import torch.distributed as dist
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        w = small(n=123_457, nd=8, r1=8, cfg=240, steps=3,
                  inject=((1, 2, wl.POS_INF, 999),))
        first, n_span, n_valid = w.span()
        states, infos = [], []
        for use_dist in (False, True):
            master, m, v, p16, ws = wl.make_state(w)
            plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
            z.zero_plan_bind(plan, 0, 8, master, m, v, p16, ws, 0)
            grads = [torch.empty(n_span, dtype=torch.float16, device="cuda") for _ in range(8)]
            inf = []
            for step in range(w.steps):
                wl.fill_grads(w, step, grads)
                if use_dist:
                    z.zero_dist_step(plan, 0, 8, grads, w.loss_scale, w.clip)
                else:
                    z.zero_shard_step(plan, 0, 8, grads, w.loss_scale, w.clip)
                inf.append(z.zero_step_result(plan).as_dict())
            states.append([f32(master), f32(m), f32(v), h16(p16)])
            infos.append(inf)
            plan.close()
        assert infos[0] == infos[1] and [x["skipped"] for x in infos[0]] == [0, 1, 0]
        for a, b in zip(*states):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("n", [300_001, 6_000_001])
def test_step_captured_in_a_cuda_graph_matches_eager_steps(n):
    # the step's launches make no host-side decision, so they can be captured once and
    # replayed; replays must give the same bits as eager calls (including an overflow
    # skip). 300,001 parameters take the one-launch step (a cooperative kernel node);
    # 6,000,001 run the reduce and update kernels with a full wave, and the capture then
    # holds the fork to the plan's second stream, its one-thread kernel and the join.
    w = small(n=n, nd=8, r1=8, cfg=250, steps=4, inject=((2, 3, wl.POS_INF, 4321),))
    first, n_span, n_valid = w.span()
    results = []
    for graph in (False, True):
        master, m, v, p16, ws = wl.make_state(w)
        plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
        z.zero_plan_bind(plan, 0, 8, master, m, v, p16, ws, 0)
        grads = [torch.empty(n_span, dtype=torch.float16, device="cuda") for _ in range(8)]
        infos = []
        if graph:
            # one ordinary call on a throw-away plan does the per-device kernel set-up
            warm = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
            wm, wmm, wv, wp, wws = wl.make_state(w)
            z.zero_plan_bind(warm, 0, 8, wm, wmm, wv, wp, wws, 0)
            wl.fill_grads(w, 0, grads)
            z.zero_shard_step(warm, 0, 8, grads, w.loss_scale, w.clip)
            torch.cuda.synchronize()
            warm.close()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                z.zero_shard_step(plan, 0, 8, grads, w.loss_scale, w.clip)
            # capture does not run the kernels; replay each step after refilling the inputs
            for step in range(w.steps):
                wl.fill_grads(w, step, grads)
                g.replay()
                torch.cuda.synchronize()
                infos.append(z.zero_step_result(plan).as_dict())
        else:
            for step in range(w.steps):
                wl.fill_grads(w, step, grads)
                z.zero_shard_step(plan, 0, 8, grads, w.loss_scale, w.clip)
                infos.append(z.zero_step_result(plan).as_dict())
        results.append((infos, [f32(master), f32(m), f32(v), h16(p16)]))
        plan.close()
    assert results[0][0] == results[1][0]
    assert [x["skipped"] for x in results[0][0]] == [0, 0, 1, 0]
    for a, b in zip(results[0][1], results[1][1]):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_two_plans_on_two_streams_concurrently():
    # plans keep separate scratch, so two steps in flight at once on different streams
    # give the same bits as each run alone
    ws_ = [small(n=400_003, nd=4, cfg=260 + k, steps=3) for k in range(2)]
    alone = []
    for w in ws_:
        r = Runner(w).run()
        assert r.exact
        alone.append([f32(t).copy() if t.dtype == torch.float32 else h16(t).copy()
                      for t in r.state[:4]])
        r.plan.close()
    plans, states, grads = [], [], []
    for w in ws_:
        st = wl.make_state(w)
        p = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
        z.zero_plan_bind(p, 0, w.nd, *st, 0)
        plans.append(p)
        states.append(st)
        grads.append([[g for g in wl.make_grads(w, s)] for s in range(w.steps)])
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in range(3):
        for k in range(2):
            with torch.cuda.stream(streams[k]):
                z.zero_shard_step(plans[k], 0, 4, grads[k][s], ws_[k].loss_scale, ws_[k].clip)
    torch.cuda.synchronize()
    for k in range(2):
        got = [f32(t) if t.dtype == torch.float32 else h16(t) for t in states[k][:4]]
        for a, b in zip(got, alone[k]):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
        plans[k].close()


@pytest.mark.parametrize("n", [400_003, 5_000_001])
def test_two_host_threads_each_with_a_plan(n):
    # one plan per host thread, stepping at the same time (the library's host code runs
    # concurrently: ctypes releases the interpreter lock); each thread's state must be the
    # bits of the same steps run alone. 400,003 parameters take the one-launch step,
    # 5,000,001 the two-kernel step with the second stream.
    import threading
    ws_ = [small(n=n, nd=4, cfg=270 + k, steps=3) for k in range(2)]
    grads = [[wl.make_grads(w, s) for s in range(w.steps)] for w in ws_]

    def run(k, out):
        w = ws_[k]
        st = wl.make_state(w)
        p = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
        z.zero_plan_bind(p, 0, w.nd, *st, 0)
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            for s in range(w.steps):
                z.zero_shard_step(p, 0, w.nd, grads[k][s], w.loss_scale, w.clip, stream)
            out[k] = z.zero_step_result(p).as_dict()
        out[k]["state"] = [f32(t).copy() if t.dtype == torch.float32 else h16(t).copy()
                           for t in st[:4]]
        p.close()

    alone = {}
    for k in range(2):
        run(k, alone)
    torch.cuda.synchronize()
    together = {}
    threads = [threading.Thread(target=run, args=(k, together)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    for k in range(2):
        assert together[k]["step"] == alone[k]["step"] == 3
        for a, b in zip(together[k]["state"], alone[k]["state"]):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_one_launch_step_boundary():
    # the one-launch step bulk-loads the state of slices up to 1024 groups of 8 per SM
    # and reads it from global memory up to 3072; the smallest span past that runs the
    # reduce and update kernels; all follow the oracle
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_pre, n_max = sms * 1024 * 8, sms * 3072 * 8
    for n, one_launch in ((n_pre, True), (n_pre + 8, True), (n_max, True), (n_max + 8, False)):
        w = small(n=n, nd=4, cfg=280 + int(one_launch), steps=2)
        r = Runner(w).run()
        assert r.exact
        ms, counts = z.zero_profile_read(r.plan)
        z.zero_profile_enable(r.plan, True)
        grads = wl.make_grads(w, 0)
        z.zero_shard_step(r.plan, 0, 4, grads, w.loss_scale, w.clip)
        ms, counts = z.zero_profile_read(r.plan, reset=True)
        assert (counts[z.PROF_STEP] == 1) == one_launch, (n, counts)
        r.plan.close()
