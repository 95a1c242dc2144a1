import ctypes
"""The C ABI of libzero without a GPU: it loads, exports every symbol include/zero.h
declares, computes the partition and accounting like the oracle, and rejects every bad
argument with the right code before any CUDA call."""
import os
import re

import pytest
import torch

import oracle
import sharded_emulated_reduce_gb300 as z

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def declared_functions():
    with open(os.path.join(ROOT, "include", "zero.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zero_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported_and_bound():
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(z._lib, n), n
    assert sorted(z.EXPORTED) == names


def test_header_constants_match_binding():
    with open(os.path.join(ROOT, "include", "zero.h")) as f:
        text = f.read()
    consts = dict(re.findall(r"#define (ZERO_\w+) \(?(-?\d+)\)?", text))
    for k, v in consts.items():
        assert getattr(z, k) == int(v), k


@pytest.mark.parametrize("n,nd,align", [(1, 1, 8), (7, 3, 8), (1023, 4, 16), (1_048_576, 4, 8),
                                        (124_439_808, 8, 128), (1_300_000_000, 16, 8),
                                        (13_000_000_000, 64, 8), (5, 256, 8)])
def test_layout_matches_oracle(n, nd, align):
    with z.zero_plan_create(n, nd, 2, align, HP) as p:
        assert z.zero_plan_layout(p) == oracle.partition(n, nd, align)
        _, s = oracle.partition(n, nd, align)
        assert z.zero_workspace_bytes(p, 0, nd) == 4 * nd * s
        assert z.zero_workspace_bytes(p, nd - 1, nd) == 4 * s


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_memory_bytes_matches_oracle(stage):
    for n, nd, align in [(7_000_000_000, 1, 8), (100_000_000_000, 64, 8), (1000, 7, 16),
                         (124_439_808, 8, 128)]:
        assert z.zero_memory_bytes(n, nd, align, stage) == oracle.memory_bytes(n, nd, align, stage)


def expect(code, fn, *args, match=None):
    with pytest.raises(z.ZeroError) as ei:
        fn(*args)
    assert ei.value.code == code, str(ei.value)
    if match:
        assert re.search(match, str(ei.value)), str(ei.value)


def test_create_rejects_bad_arguments():
    bad = [
        (0, 4, 2, 8, HP), (-1, 4, 2, 8, HP), (10, 0, 2, 8, HP), (10, 257, 2, 8, HP),
        (10, 4, 0, 8, HP), (10, 4, 4, 8, HP), (10, 4, 2, 4, HP), (10, 4, 2, 12, HP),
        (10, 4, 2, 0, HP), (10, 4, 2, 8, dict(HP, beta1=1.0)), (10, 4, 2, 8, dict(HP, beta2=-0.1)),
        (10, 4, 2, 8, dict(HP, eps=0.0)), (10, 4, 2, 8, dict(HP, lr=float("nan"))),
        (10, 4, 2, 8, dict(HP, weight_decay=-1.0)), (10, 4, 2, 8, dict(HP, lr=float("inf"))),
        (2**40, 64, 3, 8, HP),  # Np * nd^2 >= 2^47
    ]
    for args in bad:
        expect(z.ZERO_EINVAL, z.zero_plan_create, *args)
    assert z.zero_last_error()


def test_bind_rejects_null_and_unaligned_pointers():
    with z.zero_plan_create(100, 4, 2, 8, HP) as p:
        good = 0x10000
        expect(z.ZERO_EINVAL, z.zero_plan_bind, p, 0, 4, 0, good, good, good, good)
        expect(z.ZERO_EINVAL, z.zero_plan_bind, p, 0, 4, good, good, good, good, 0)
        for i in range(5):
            ptrs = [good] * 5
            ptrs[i] = good + 8
            expect(z.ZERO_EALIGN, z.zero_plan_bind, p, 0, 4, *ptrs)
        expect(z.ZERO_EINVAL, z.zero_plan_bind, p, 0, 4, *([good] * 5), -1)
        for r0, r1 in [(-1, 2), (0, 5), (2, 2), (3, 1)]:
            expect(z.ZERO_EINVAL, z.zero_plan_bind, p, r0, r1, *([good] * 5))


def test_step_rejects_bad_arguments_before_touching_the_device():
    with z.zero_plan_create(100, 4, 2, 8, HP) as p:
        good = [0x10000 + 0x1000 * k for k in range(4)]
        for r0, r1 in [(-1, 2), (0, 5), (2, 2)]:
            expect(z.ZERO_EINVAL, z.zero_shard_step, p, r0, r1, good, 1.0, 0.0, 0)
        expect(z.ZERO_EINVAL, z.zero_shard_step, p, 0, 4, good[:3] + [0], 1.0, 0.0, 0)
        expect(z.ZERO_EALIGN, z.zero_shard_step, p, 0, 4, good[:3] + [good[3] + 2], 1.0, 0.0, 0)
        for ls in [0.0, -1.0, float("inf"), float("nan")]:
            expect(z.ZERO_EINVAL, z.zero_shard_step, p, 0, 4, good, ls, 0.0, 0)
        expect(z.ZERO_EINVAL, z.zero_shard_step, p, 0, 4, good, 1.0, float("nan"), 0)
        # all arguments valid, but nothing is bound
        expect(z.ZERO_EUNBOUND, z.zero_shard_step, p, 0, 4, good, 1.0, 0.0, 0)
        expect(z.ZERO_EUNBOUND, z.zero_shard_reduce, p, 0, 4, good, 0)
        expect(z.ZERO_EUNBOUND, z.zero_shard_update, p, 0, 4, 1.0, 1.0, 0)
        expect(z.ZERO_EINVAL, z.zero_shard_update, p, 0, 4, 0.0, 1.0, 0)
        expect(z.ZERO_EUNBOUND, z.zero_step_result, p)
        expect(z.ZERO_EUNBOUND, z.zero_shard_stats, p)


def test_gather_rejects_bad_arguments():
    with z.zero_plan_create(100, 4, 3, 8, HP) as p:
        shards = [0x10000 + 0x1000 * k for k in range(4)]
        dst = [0x40000, 0x50000]
        expect(z.ZERO_EINVAL, z.zero_gather_layers, p, [0], shards, [], 0)          # no layer
        expect(z.ZERO_EINVAL, z.zero_gather_layers, p, [-1, 50, 100], shards, dst, 0)
        expect(z.ZERO_EINVAL, z.zero_gather_layers, p, [0, 60, 50], shards, dst, 0)
        expect(z.ZERO_EINVAL, z.zero_gather_layers, p, [0, 50, 101], shards, dst, 0)  # > N
        expect(z.ZERO_EINVAL, z.zero_gather_layers, p, [0, 50, 100], shards, [0x40000, 0], 0)
        expect(z.ZERO_EALIGN, z.zero_gather_layers, p, [0, 50, 100], shards, [0x40001, 0x50000], 0)
        expect(z.ZERO_EINVAL, z.zero_gather_layers, p, [0, 50, 100], shards[:3] + [0], dst, 0)
        expect(z.ZERO_EALIGN, z.zero_gather_layers, p, [0, 50, 100], shards[:3] + [shards[3] + 1],
               dst, 0)
        # the layer-by-layer form: the same checks, plus the event array itself
        ev = [0x70000, 0]
        expect(z.ZERO_EINVAL, z.zero_gather_layers_events, p, [0, 60, 50], shards, dst, ev, 0)
        expect(z.ZERO_EALIGN, z.zero_gather_layers_events, p, [0, 50, 100], shards,
               [0x40001, 0x50000], ev, 0)
        expect(z.ZERO_EINVAL, z.zero_gather_layers_events, p, [0, 50, 100], shards, dst, [0], 0)
        offs = (z._I64 * 3)(0, 50, 100)
        rc = z._lib.zero_gather_layers_events(p, offs, 2, z._ptrs(shards), z._ptrs(dst), None, 0)
        assert rc == z.ZERO_EINVAL and "layer_done" in z.zero_last_error()


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_calls_report_cuda_errors_without_a_gpu():
    with z.zero_plan_create(100, 4, 2, 8, HP) as p:
        expect(z.ZERO_ECUDA, z.zero_plan_bind, p, 0, 4, *([0x10000] * 5))
        expect(z.ZERO_ECUDA, z.zero_gather_layers, p, [0, 100],
               [0x10000 + 0x1000 * k for k in range(4)], [0x40000], 0)


def test_profile_calls_on_a_fresh_plan():
    with z.zero_plan_create(100, 4, 2, 8, HP) as p:
        z.zero_profile_enable(p, True)
        ms, n = z.zero_profile_read(p, reset=True)
        assert ms == [0.0] * z.ZERO_PROF_KINDS and n == [0] * z.ZERO_PROF_KINDS


def test_destroyed_plan_is_refused_by_the_binding():
    p = z.zero_plan_create(100, 4, 2, 8, HP)
    p.close()
    with pytest.raises(Exception, match="destroyed"):
        z.zero_plan_layout(p)


def test_scaler_and_state_calls_validate_before_touching_the_device():
    with z.zero_plan_create(100, 4, 2, 8, HP) as p:
        for kw in [dict(scale=0.0, growth_interval=10), dict(scale=float("inf"), growth_interval=1),
                   dict(growth_factor=0.5, growth_interval=1), dict(backoff_factor=0.0, growth_interval=1),
                   dict(backoff_factor=1.5, growth_interval=1), dict(growth_interval=-1),
                   dict(good_steps=-1, growth_interval=5)]:
            expect(z.ZERO_EINVAL, lambda: z.zero_plan_set_scaler(p, **kw))
        expect(z.ZERO_EUNBOUND, lambda: z.zero_plan_set_scaler(p, growth_interval=100))
        expect(z.ZERO_EUNBOUND, z.zero_loss_scale_ptr, p)
        expect(z.ZERO_EUNBOUND, z.zero_plan_get_state, p)
        st = z.zero_plan_state()
        st.step = -1
        expect(z.ZERO_EINVAL, z.zero_plan_set_state, p, st)
        st.step = 3
        expect(z.ZERO_EUNBOUND, z.zero_plan_set_state, p, st)


def test_selftest_rejects_bad_poll_counts():
    for polls in (0, 2**24 + 1):
        expect(z.ZERO_EINVAL, z.zero_selftest_wait, polls)
        expect(z.ZERO_EINVAL, z.zero_selftest_grid_barrier, polls)


def test_bounds_report_of_the_normal_build():
    # the normal build compiles no checks: it reports them off, with no fault, and needs
    # no device to say so; NULL outputs are rejected
    assert z.zero_bounds_check() == {"enabled": 0, "site": 0, "offset": 0}
    lib = z.lib()
    out = z._I32()
    assert lib.zero_bounds_check(0, None, ctypes.byref(out), None) == z.ZERO_EINVAL


def test_gather_status_without_a_gather_is_zero():
    with z.zero_plan_create(100, 4, 3, 8, HP) as p:
        assert z.zero_gather_status(p) == 0
