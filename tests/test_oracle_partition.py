"""Pins of the oracle's partitioner and memory accounting against the pages and brute force.

Partition: ZeRO partitions the model states across ranks ("ZeRO" method entry,
description). Accounting: ZeRO explainer, "The 16 Bytes per Parameter Audit", Chapter 01
and Chapter 02, stage table.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_padded(n, nd, align):
    np_ = n
    while np_ % (nd * align):
        np_ += 1
    return np_


@pytest.mark.parametrize("align", [8, 16, 128])
def test_partition_matches_brute_force(align):
    for n in range(1, 301):
        for nd in range(1, 10):
            np_, s = oracle.partition(n, nd, align)
            assert np_ == brute_padded(n, nd, align)
            assert s * nd == np_
            assert s % align == 0          # every shard starts on an aligned element
            assert np_ - n < nd * align    # padding is less than one unit


def test_partition_large_shapes():
    # sizes of the workloads: GPT-2-small flat buffer with 128-element alignment, 1.3B,
    # the 7B and 13B per-rank shards
    assert oracle.partition(124_439_808, 8, 128) == (124_440_576, 15_555_072)
    assert oracle.partition(1_048_576, 4, 8) == (1_048_576, 262_144)
    assert oracle.partition(1_300_000_000, 16, 8) == (1_300_000_000, 81_250_000)
    assert oracle.partition(7_000_000_000, 8, 8) == (7_000_000_000, 875_000_000)
    assert oracle.partition(13_000_000_000, 64, 8) == (13_000_000_000, 203_125_000)
    for n, nd, al in [(124_439_808, 8, 128), (2**40 + 3, 64, 8)]:
        np_, s = oracle.partition(n, nd, al)
        assert np_ == brute_padded(n, nd, al) if np_ - n < 10**6 else True
        assert np_ >= n and np_ % (nd * al) == 0 and s == np_ // nd


def test_partition_rejects_bad_input():
    for args in [(0, 4, 8), (-5, 4, 8), (10, 0, 8), (10, 4, 0)]:
        with pytest.raises(ValueError):
            oracle.partition(*args)


def test_shards_concatenate_to_flat_buffer():
    rng = np.random.default_rng(0)
    for n, nd, align in [(1, 1, 8), (7, 3, 8), (1023, 4, 16), (5000, 9, 128), (64, 8, 8)]:
        np_, s = oracle.partition(n, nd, align)
        flat = np.zeros(np_, dtype=np.uint16)
        flat[:n] = rng.integers(0, 65536, n, dtype=np.uint16)
        shards = [flat[r * s:(r + 1) * s].copy() for r in range(nd)]
        assert all(sh.size == s for sh in shards)
        assert np.array_equal(np.concatenate(shards), flat)
        assert not flat[n:].any()


def load_accounting():
    with open(os.path.join(GOLDEN, "accounting.json")) as f:
        return json.load(f)


def test_accounting_printed_totals():
    g = load_accounting()
    for key in ("model_7B", "model_100B"):
        case = g[key]
        got = oracle.memory_bytes(case["params"], 1, 8, 0)
        assert got == case["bytes"]
        # per-parameter replicated bytes are the audit's 16
        assert got // case["params"] == g["bytes_per_param_replicated"]["value"]


def test_accounting_stage_ratios_tend_to_the_printed_limits():
    g = load_accounting()
    n = 2**40  # divisible by every Nd * align below, so padding does not blur the ratio
    prev = {1: 0.0, 2: 0.0}
    for nd in [2, 4, 16, 64, 1024, 2**16, 2**20]:
        base = oracle.memory_bytes(n, nd, 8, 0)
        for stage in (1, 2):
            r = base / oracle.memory_bytes(n, nd, 8, stage)
            assert r > prev[stage]          # monotone in Nd
            assert r < g["stage_reduction"][str(stage)]["limit"]
            prev[stage] = r
        # ZeRO-3: per-rank bytes are exactly 1/Nd of the replicated bytes
        assert oracle.memory_bytes(n, nd, 8, 3) * nd == base
    for stage in (1, 2):
        limit = g["stage_reduction"][str(stage)]["limit"]
        assert abs(prev[stage] - limit) / limit < 1e-4


def test_accounting_at_64_ranks():
    n, nd = 13_000_000_000, 64
    base = oracle.memory_bytes(n, nd, 8, 0)
    r1 = base / oracle.memory_bytes(n, nd, 8, 1)
    r2 = base / oracle.memory_bytes(n, nd, 8, 2)
    r3 = base / oracle.memory_bytes(n, nd, 8, 3)
    # 16 / (4 + 12/64), 16 / (2 + 14/64), 64
    assert r1 == pytest.approx(16 / (4 + 12 / 64), rel=1e-12)
    assert r2 == pytest.approx(16 / (2 + 14 / 64), rel=1e-12)
    assert r3 == 64.0


def test_accounting_rejects_bad_stage():
    assert oracle.memory_bytes(100, 4, 8, 4) == -1
    assert oracle.memory_bytes(0, 4, 8, 1) == -1
