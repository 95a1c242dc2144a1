"""GPU: a span split across two processes, through the library's own split-step calls.

ZeRO's reduce-scatter leaves each data-parallel process with the summed gradients of its
own partition; the global norm and the overflow flag then need one exchange across the
processes (ZeRO explainer, Chapter 02, ZeRO-3 item "reduce-scatter after backward").
Here two processes on the one GPU each own half of the logical ranks of one flat
buffer. Each runs zero_shard_reduce on its half, copies the plan's 8 exchange words to
the host, sums them with the other process over gloo, writes the sum back and runs
zero_shard_update. No kernel waits on the other process: the only wait is the host-side
all-reduce between two launches. The halves' results must be bit-identical to one
process stepping the whole span with zero_shard_step on the same inputs, including a
step whose +inf sits in only one process's half and must make both skip.
"""
import dataclasses
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

STEPS = 3


def workload(n):
    from synth import workloads as wl
    # the +inf of the second step lies in the second process's half only
    return wl.Workload("split", cfg=600, n=n, nd=8, align=8, stage=2, r0=0, r1=8,
                       loss_scale=65536.0, grad_sigma=1e-3, clip=1.0, steps=STEPS,
                       m_sigma=1e-3, v_sigma=1e-6, inject=((1, 6, wl.POS_INF, 3 * n // 4),))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def host_state(master, m, v, p16):
    return (master.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy(),
            p16.cpu().view(torch.int16).numpy().view(np.uint16))


def worker(rank, world, port, n, q):
    import torch.distributed as dist

    import sharded_emulated_reduce_gb300 as z
    from synth import workloads as wl
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        w0 = workload(n)
        r0, r1 = z.rank_ranges(w0.nd, world)[rank]
        w = dataclasses.replace(w0, r0=r0, r1=r1)
        master, m, v, p16, ws = wl.make_state(w)
        plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
        z.zero_plan_bind(plan, r0, r1, master, m, v, p16, ws, 0)
        words = z.stats_tensor(plan)
        stream = torch.cuda.current_stream()
        infos = []
        for step in range(STEPS):
            grads = wl.make_grads(w, step)
            z.zero_shard_reduce(plan, r0, r1, grads, stream)
            host = words.cpu()                # waits for the reduce
            dist.all_reduce(host)             # the exchange: an exact integer sum
            words.copy_(host)
            z.zero_shard_update(plan, r0, r1, w.loss_scale, w.clip, stream)
            infos.append(z.zero_step_result(plan).as_dict())
        q.put((rank, infos, host_state(master, m, v, p16)))
        plan.close()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("n", [2_000_003, 40_000_000])
def test_two_processes_split_the_span_bit_identically(n):
    import sharded_emulated_reduce_gb300 as z
    from synth import workloads as wl
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, world, port, n, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(world):
            rank, infos, state = q.get(timeout=600)
            got[rank] = (infos, state)
    finally:
        for p in procs:
            p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)

    # one process stepping the whole span on the same inputs
    w = workload(n)
    master, m, v, p16, ws = wl.make_state(w)
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, 0, w.nd, master, m, v, p16, ws, 0)
    ref = []
    for step in range(STEPS):
        grads = wl.make_grads(w, step)
        z.zero_shard_step(plan, 0, w.nd, grads, w.loss_scale, w.clip)
        ref.append(z.zero_step_result(plan).as_dict())
    whole = host_state(master, m, v, p16)
    plan.close()

    assert [x["skipped"] for x in ref] == [0, 1, 0]
    _, s = w.layout()
    for rank in range(world):
        infos, state = got[rank]
        for a, b in zip(infos, ref):
            for k in ("overflow", "skipped", "step", "sum_sq", "global_norm", "clip_coef",
                      "scale", "bc1", "bc2", "status"):
                assert a[k] == b[k], (rank, k, a[k], b[k])
        r0, r1 = z.rank_ranges(w.nd, world)[rank]
        sl = slice(r0 * s, r1 * s)
        for x, y in zip(state, whole):
            x_bits = x.view(np.uint32) if x.dtype == np.float32 else x
            y_bits = y[sl].view(np.uint32) if y.dtype == np.float32 else y[sl]
            assert np.array_equal(x_bits, y_bits), rank


def test_bench_line_from_two_processes():
    # the bench's multi-process path (process group, barriers, max over processes, rank
    # 0's single line), rehearsed with two processes sharing the one GPU over gloo: the
    # 1M workload's four logical ranks split over the two (strong scaling)
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, ZERO_BENCH_BACKEND="gloo")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--gpus", "2", "--workload", "zero2_tiny_1m_nd4", "--steps", "5", "--warmup", "3",
           "--cpu-seconds", "0"]
    out = subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["scaling"] == "strong" and d["value"] > 0
    assert d["config"]["workload"] == "zero2_tiny_1m_nd4"
    assert d["e2e"]["value"] > 0 and d["gather"]["value"] > 0
    assert d["last_step"]["skipped"] == 0
