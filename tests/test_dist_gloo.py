"""The exchange step of a span split across processes, on CPU with two gloo ranks.

Each process owns half of the logical ranks (rank_ranges), computes its span's
statistics with the oracle in the exchange-buffer format (stats_words), and the
processes sum the words with an all-reduce. The summed words must decode to exactly the
statistics of the whole buffer, so the step's scalars (norm, clip coefficient, skip) are
the same as in one process; the per-element update then matches the unsplit step.
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth
import sharded_emulated_reduce_gb300 as z


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def grads_for(n, nd, seed, inject=None):
    out = []
    for k in range(nd):
        key = synth.stream_key(seed, synth.GRAD, 50, 0, k)
        g = synth.values_f16(key, 1e-2 * 65536, 0, n)
        out.append(g)
    if inject is not None:
        out[inject[0]][inject[1]] = 0x7C00
    return out


def worker(rank, world, port, n, nd, inject, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch
    np_, s = oracle.partition(n, nd, 8)
    r0, r1 = z.rank_ranges(nd, world)[rank]
    a, b = r0 * s, min(r1 * s, n)
    g = grads_for(np_, nd, 1, inject)
    gsum = oracle.reduce([x[a:b] for x in g])
    bad, ss = oracle.stats(gsum)
    words = torch.tensor(z.stats_words(bad, ss), dtype=torch.int64)
    dist.all_reduce(words)
    q.put((rank, words.tolist()))
    dist.destroy_process_group()


@pytest.mark.parametrize("inject", [None, (3, 777)])
def test_two_process_exchange_is_exact(inject):
    n, nd, world = 50_003, 8, 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, world, port, n, nd, inject, q))
             for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == got[1]
    np_, s = oracle.partition(n, nd, 8)
    g = grads_for(np_, nd, 1, inject)
    bad, ss = oracle.stats(oracle.reduce([x[:n] for x in g]))
    assert z.stats_decode(got[0]) == (bad, ss)
    hp = oracle.Hyper()
    whole = oracle.scalars(bad, ss, 65536.0, 1.0, hp, 0)
    split = oracle.scalars(*z.stats_decode(got[0]), 65536.0, 1.0, hp, 0)
    assert (whole.skipped, whole.ss, whole.norm, whole.s) == (split.skipped, split.ss, split.norm,
                                                              split.s)
    assert whole.skipped == (inject is not None)


def test_rank_ranges():
    assert z.rank_ranges(8, 1) == [(0, 8)]
    assert z.rank_ranges(8, 2) == [(0, 4), (4, 8)]
    assert z.rank_ranges(64, 8)[-1] == (56, 64)
    with pytest.raises(ValueError):
        z.rank_ranges(8, 3)


def test_stats_words_roundtrip_and_limb_sums():
    rng = np.random.default_rng(0)
    for _ in range(100):
        parts = [(int(rng.integers(0, 5)), int(rng.integers(0, 2**62)) * int(rng.integers(1, 2**60)))
                 for _ in range(8)]
        summed = [sum(col) for col in zip(*[z.stats_words(b, s) for b, s in parts])]
        assert all(0 <= w < 2**63 for w in summed)
        assert z.stats_decode(summed) == (sum(b for b, _ in parts), sum(s for _, s in parts))
