"""GPU: the bounded-wait failure path, exercised without faulting or hanging the GPU.

A kernel waits on a shared-memory barrier that nothing completes, with a short poll
limit; it must give up, report it, and leave the context usable for a normal step."""
import time

import pytest

import sharded_emulated_reduce_gb300 as z
from synth import workloads as wl

from parity import Runner

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_and_reports():
    for polls in (1, 64, 4096):
        t0 = time.perf_counter()
        assert z.zero_selftest_wait(polls) == 1
        assert time.perf_counter() - t0 < 5.0


def test_context_stays_usable_after_an_expired_wait():
    assert z.zero_selftest_wait(1000) == 1
    w = wl.Workload("after_wait", cfg=600, n=50_001, nd=4, align=8, stage=2, r0=0, r1=4,
                    loss_scale=1024.0, grad_sigma=1e-3, clip=1.0, steps=2)
    r = Runner(w).run()
    assert r.exact and all(x["status"] == 0 for x in r.results)
    assert z.zero_gather_status(r.plan) == 0


def test_grid_barrier_is_met_with_exact_sums_when_every_cta_arrives():
    for _ in range(3):  # the probe's words start from zero every run
        assert z.zero_selftest_grid_barrier(1 << 16, skip_one=False) == 0


def test_grid_barrier_gives_up_when_a_cta_never_arrives():
    for polls in (1, 64, 4096):
        t0 = time.perf_counter()
        assert z.zero_selftest_grid_barrier(polls, skip_one=True) == 1
        assert time.perf_counter() - t0 < 5.0
    # the context stays usable: a one-launch step (it uses the same barrier) afterwards
    w = wl.Workload("after_barrier", cfg=601, n=50_001, nd=4, align=8, stage=2, r0=0, r1=4,
                    loss_scale=1024.0, grad_sigma=1e-3, clip=1.0, steps=2)
    r = Runner(w).run()
    assert r.exact and all(x["status"] == 0 for x in r.results)
