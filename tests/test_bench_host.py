"""Host-side pieces of the benchmark: the chunked, threaded CPU sample generator and the
oracle's step partitioned over host threads (the all-core CPU baseline). Both must give
exactly what the single-threaded forms give."""
import numpy as np

import bench
import oracle
import synth
from synth import workloads as wl

W = wl.WORKLOADS["gpt2_small_flat_nd8"]


def test_chunked_sample_equals_direct_generation():
    n = 2 * bench.GEN_CHUNK + 4104  # three chunks, the last one ragged
    grads, master, m, v, p16 = bench.cpu_sample(W, n, threads=4)
    first = W.span()[0]
    assert np.array_equal(master, synth.values_f32(wl.key(W, synth.MASTER), W.master_sigma,
                                                   first, n))
    g = synth.values_f16(wl.key(W, synth.GRAD, 1, 5), W.grad_sigma * W.loss_scale, first, n)
    assert np.array_equal(grads[1][5], g)
    assert np.array_equal(p16, master.astype(np.float16).view(np.uint16))
    assert len(grads) == 2 and all(len(gs) == W.nd for gs in grads)


def _state(sample):
    grads, master, m, v, p16 = sample
    return grads, master.copy(), m.copy(), v.copy(), p16.copy()


def test_partitioned_oracle_is_bit_identical_to_one_step():
    n = 100_024  # a multiple of 8, not of the 64-element slice granularity
    sample = bench.cpu_sample(W, n, threads=2)
    hp = oracle.Hyper(**W.hparams())
    g1, ma, ma_m, ma_v, ma_p = _state(sample)
    g2, mb, mb_m, mb_v, mb_p = _state(sample)
    clip = 0.25  # below the sample's norm (about 0.9), so the clip is active
    par = bench.PartitionedOracle(n, 5)
    assert par.threads == 5
    ta = tb = 0
    for i in range(3):
        a = oracle.step(g1[i % 2], ma, ma_m, ma_v, ma_p, W.loss_scale, clip, hp, ta)
        b = par.step(g2[i % 2], mb, mb_m, mb_v, mb_p, W.loss_scale, clip, hp, tb)
        ta, tb = a.step, b.step
        for f in ("overflow", "skipped", "step", "ss", "norm", "clip_coef", "s", "bc1", "bc2"):
            assert getattr(a, f) == getattr(b, f), (i, f)
        assert a.clip_coef < 1.0
    for x, y in ((ma, mb), (ma_m, mb_m), (ma_v, mb_v), (ma_p, mb_p)):
        assert np.array_equal(x.view(np.uint32) if x.dtype == np.float32 else x,
                              y.view(np.uint32) if y.dtype == np.float32 else y)
    # an inf in the last slice makes the whole step skip, as in the single-threaded step
    bad = [c.copy() for c in g2[0]]
    bad[3][n - 5] = 0x7C00
    before = mb.copy()
    b = par.step(bad, mb, mb_m, mb_v, mb_p, W.loss_scale, clip, hp, tb)
    assert b.overflow == 1 and b.skipped == 1 and b.step == tb
    assert np.array_equal(before, mb)
    par.close()


def test_all_core_sample_is_bounded():
    for name in ("gpt2_small_flat_nd8", "zero3_13b_rank0_nd64"):
        w = wl.WORKLOADS[name]
        n = bench.all_core_sample_size(w, 72)
        assert n % 8 == 0 and n <= w.span()[2]
        assert n * bench.sample_bytes_per_param(w) <= bench.SAMPLE_BYTES


def test_gather_cpu_baseline_runs_on_a_scaled_layout():
    w = wl.WORKLOADS["zero3_1p3b_rank0_nd64"]
    c = bench.gather_cpu_rate(w, 0.05)
    assert c["kind"] == "oracle" and c["value"] > 0 and 1 <= c["cores"] <= len(w.layers) - 1
    assert f"{len(w.layers) - 1} layers" in c["sample"]
