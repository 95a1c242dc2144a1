"""GPU parity at the workloads' full sizes, in the launch configuration the bench times.

Every element of every output is compared on every step: the oracle's step runs over
slices of the span on all host threads (bit-identical to one oracle step), fed with the
same gradient bytes, and the GPU's master weights, moments, fp16 parameters and fp32 rank
sums are compared with it in full (bit for bit where they agree, else at the 1e-6 / 1 ulp
bar), as are the overflow flag, skip decision, step counter and exact sum of squares.
The largest case, the 1.3B buffer with 16 ranks, holds about 70 GB of host memory. The
ZeRO-3 gather is checked in full against slices of the shards and on sampled elements
against the oracle's index map, for the workload's layer boundaries and for boundaries
moved off the shards' 16-byte alignment.
"""
import numpy as np
import pytest
import torch

import oracle
import sharded_emulated_reduce_gb300 as z
from synth import workloads as wl

from parity import Runner, h16

pytestmark = pytest.mark.gpu


def test_gpt2_small_flat_nd8_all_steps():
    w = wl.WORKLOADS["gpt2_small_flat_nd8"]
    r = Runner(w, mode="full_parallel").run()
    assert len(r.results) == w.steps
    assert all(x["skipped"] == 0 for x in r.results)
    assert all(x["clip_coef"] < 1.0 for x in r.results)  # clipping is active here
    assert r.exact
    # the ZeRO-1/2 parameter all-gather after the step: the Nd fp16 shards (rank 0's is the
    # step's output, the others seeded) into one flat buffer, as the bench's full-buffer
    # gather times it; the padding of the last shard is not copied
    _, s = w.layout()
    shards = wl.make_shards(w, r.state[3][:s])
    flat = torch.empty(w.n, dtype=torch.float16, device="cuda")
    z.zero_gather_layers(r.plan, [0, w.n], shards, [flat])
    torch.cuda.synchronize()
    assert z.zero_gather_status(r.plan) == 0
    for k in range(w.nd):
        hi = min(w.n, (k + 1) * s)
        assert torch.equal(flat[k * s:hi], shards[k][:hi - k * s]), k


def test_flat_1p3b_nd16_overflow_skip():
    w = wl.WORKLOADS["flat_1p3b_nd16_inf"]
    r = Runner(w, mode="full_parallel").run()  # all 8 steps
    assert [x["skipped"] for x in r.results] == [0, 0, 1, 0, 0, 0, 0, 0]
    assert [x["step"] for x in r.results] == [1, 2, 2, 3, 4, 5, 6, 7]
    assert r.exact


def test_zero2_7b_rank0_nd8():
    w = wl.WORKLOADS["zero2_7b_rank0_nd8"]
    r = Runner(w, mode="full_parallel").run()  # all 5 steps
    assert all(x["skipped"] == 0 for x in r.results)
    assert r.exact


def test_zero3_13b_rank0_nd64_step_and_gather():
    w = wl.WORKLOADS["zero3_13b_rank0_nd64"]
    r = Runner(w, mode="full_parallel").run()  # all 5 steps
    assert r.exact
    master, m, v, p16, ws = r.state
    del master, m, v, ws
    torch.cuda.empty_cache()
    _, s = w.layout()
    shards = wl.make_shards(w, p16)
    offs = list(w.layers)
    dst = [torch.empty(offs[l + 1] - offs[l], dtype=torch.float16, device="cuda")
           for l in range(len(offs) - 1)]
    z.zero_gather_layers(r.plan, offs, shards, dst)
    torch.cuda.synchronize()
    # every layer equals the matching slices of the shards (plain slicing of the inputs)
    for l in range(len(offs) - 1):
        a, b = offs[l], offs[l + 1]
        rr = a // s
        pos = a
        while pos < b:
            hi = min(b, (rr + 1) * s)
            assert torch.equal(dst[l][pos - a:hi - a], shards[rr][pos - rr * s:hi - rr * s]), l
            pos = hi
            rr += 1
    # sampled elements against the oracle's index arithmetic
    rng = np.random.default_rng(5)
    for l in [0, 1, 19, 38, 39]:
        n_l = offs[l + 1] - offs[l]
        js = np.unique(np.concatenate([rng.integers(0, n_l, 512), [0, n_l - 1]]))
        got = h16(dst[l][torch.as_tensor(js, device="cuda")])
        for j, g in zip(js.tolist(), got.tolist()):
            rank, off = oracle.gather_source(s, offs[l] + j)
            assert g == int(h16(shards[rank][off:off + 1])[0])
    # the same shards with every interior layer boundary moved by 3 elements (the bench's
    # --layer-shift 3): layers 1..39 are misaligned against the shards modulo 16 bytes and
    # go through the realigning kernel
    del dst
    torch.cuda.empty_cache()
    offs3 = [offs[0]] + [o + 3 for o in offs[1:-1]] + [offs[-1]]
    dst3 = [torch.empty(offs3[l + 1] - offs3[l], dtype=torch.float16, device="cuda")
            for l in range(len(offs3) - 1)]
    z.zero_gather_layers(r.plan, offs3, shards, dst3)
    torch.cuda.synchronize()
    assert z.zero_gather_status(r.plan) == 0
    for l in range(len(offs3) - 1):
        a, b = offs3[l], offs3[l + 1]
        rr = a // s
        pos = a
        while pos < b:
            hi = min(b, (rr + 1) * s)
            assert torch.equal(dst3[l][pos - a:hi - a], shards[rr][pos - rr * s:hi - rr * s]), l
            pos = hi
            rr += 1
    for l in [0, 1, 20, 39]:
        n_l = offs3[l + 1] - offs3[l]
        js = np.unique(np.concatenate([rng.integers(0, n_l, 512), [0, 1, 2, n_l - 1]]))
        got = h16(dst3[l][torch.as_tensor(js, device="cuda")])
        for j, g in zip(js.tolist(), got.tolist()):
            rank, off = oracle.gather_source(s, offs3[l] + j)
            assert g == int(h16(shards[rank][off:off + 1])[0])
