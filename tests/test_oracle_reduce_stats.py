"""Pins of the oracle's rank-order reduction, overflow flag and sum of squares.

The reduction is the arithmetic of the reduce-scatter (ZeRO explainer, Chapter 02,
ZeRO-3 item: reduce-scatter after backward); the flag and the norm are what mixed
precision and global-norm clipping need (ZeRO explainer, "The mixed-precision era").
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_f16(rng, n, scale=1.0):
    return (rng.standard_normal(n) * scale).astype(np.float16).view(np.uint16)


def exact_units(h):
    """fp16 bit patterns -> exact integers in units of 2^-24 (Python ints via float64)."""
    f = h.view(np.float16).astype(np.float64)
    return f * 2.0**24  # exact: fp16 values are integer multiples of 2^-24 below 2^16


def test_rank_order_golden():
    with open(os.path.join(GOLDEN, "rank_order.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        contrib = [np.array([b], dtype=np.uint16) for b in case["contrib_f16_bits"]]
        got = oracle.reduce(contrib)[0]
        if case["expected_f32"] == "nan":
            assert math.isnan(got)
        else:
            assert got == np.float32(case["expected_f32"])
            if "expected_sign_bit" in case:
                assert (np.float32(got).view(np.uint32) >> 31) == case["expected_sign_bit"]


def test_single_rank_is_exact():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.reduce([h])
    ref = h.view(np.float16).astype(np.float32)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin] + np.float32(0.0))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_two_ranks_equal_rounded_exact_sum():
    rng = np.random.default_rng(2)
    n = 1 << 18
    a = rng.integers(0, 65536, n, dtype=np.uint64).astype(np.uint16)
    b = rng.integers(0, 65536, n, dtype=np.uint64).astype(np.uint16)
    got = oracle.reduce([a, b])
    fa, fb = a.view(np.float16).astype(np.float64), b.view(np.float16).astype(np.float64)
    fin = np.isfinite(fa) & np.isfinite(fb)
    # the exact sum of two fp16 values is an integer multiple of 2^-24 below 2^17, so it
    # is exact in float64; one rounding to fp32 is then the correctly rounded sum
    exact = exact_units(a[fin]) + exact_units(b[fin])
    ref = (exact * 2.0**-24).astype(np.float32)
    assert np.array_equal(got[fin], ref)


def test_many_ranks_within_recursive_summation_bound():
    rng = np.random.default_rng(3)
    nd, n = 64, 1 << 14
    contrib = [rand_f16(rng, n, 50.0) for _ in range(nd)]
    got = oracle.reduce(contrib).astype(np.float64)
    units = np.stack([exact_units(c) for c in contrib])
    exact = units.sum(axis=0) * 2.0**-24  # int-valued float64 sums stay exact here
    mag = np.abs(units).sum(axis=0) * 2.0**-24
    bound = (nd - 1) * 2.0**-24 * mag * (1 + 1e-6)
    assert np.all(np.abs(got - exact) <= bound)
    assert np.any(got != exact)  # the bound is not vacuous: rounding did happen


def test_padding_sums_to_zero_even_with_garbage():
    rng = np.random.default_rng(4)
    n, nv = 100, 61
    contrib = [rand_f16(rng, n) for _ in range(3)]
    contrib[1][nv:] = 0x7C00  # +inf in the padding only
    got = oracle.reduce(contrib, n_valid=nv)
    assert np.all(got[nv:] == 0)
    assert np.all(np.isfinite(got[:nv]))


def test_sum_of_squares_is_exactly_rounded():
    rng = np.random.default_rng(5)
    for nd, n, scale in [(1, 1000, 1.0), (4, 4096, 1e3), (8, 10000, 1e-3), (16, 333, 6e4)]:
        contrib = [rand_f16(rng, n, scale) for _ in range(nd)]
        g = oracle.reduce(contrib)
        if not np.all(np.isfinite(g)):
            continue
        bad, ss = oracle.stats(g)
        assert bad == 0
        sc = oracle.scalars(bad, ss, 1.0, 0.0, oracle.Hyper(), 0)
        # each fp32 square is exact in float64; fsum is the correctly rounded exact sum
        ref = math.fsum(float(x) * float(x) for x in g.astype(np.float64))
        assert sc.ss == ref
        # and the integer form really is integer
        k = g.astype(np.float64) * 2.0**24
        assert np.all(np.floor(k) == k)


def test_norm_matches_torch_float64():
    rng = np.random.default_rng(6)
    contrib = [rand_f16(rng, 50000, 1e-3 * 1024) for _ in range(4)]
    g = oracle.reduce(contrib)
    bad, ss = oracle.stats(g)
    sc = oracle.scalars(bad, ss, 1024.0, 0.0, oracle.Hyper(), 0)
    ref = torch.linalg.vector_norm(torch.from_numpy(g.astype(np.float64))).item() / 1024.0
    assert sc.norm == pytest.approx(ref, rel=1e-13)


@pytest.mark.parametrize("where", ["first", "middle", "last"])
@pytest.mark.parametrize("value", [0x7C00, 0xFC00, 0x7E00, "both"])
def test_overflow_flag_brute_force(where, value):
    rng = np.random.default_rng(7)
    n, nd = 999, 5
    contrib = [rand_f16(rng, n) for _ in range(nd)]
    i = {"first": 0, "middle": n // 2, "last": n - 1}[where]
    if value == "both":
        contrib[0][i] = 0x7C00
        contrib[nd - 1][i] = 0xFC00
    else:
        contrib[nd - 1][i] = value
    g = oracle.reduce(contrib)
    bad, _ = oracle.stats(g)
    fl = np.stack([c.view(np.float16).astype(np.float32) for c in contrib])
    brute = int(np.sum(~np.all(np.isfinite(fl), axis=0) | ~np.isfinite(fl.sum(axis=0))))
    assert bad == brute == 1
    sc = oracle.scalars(bad, 0, 1.0, 1.0, oracle.Hyper(), 7)
    assert sc.overflow == 1 and sc.skipped == 1 and sc.step == 7 and math.isinf(sc.norm)


def test_synthetic_gradients_sum_without_fp32_overflow():
    # the largest finite fp16 sum of 64 ranks stays finite in fp32
    big = np.full(1, 0x7BFF, dtype=np.uint16)
    g = oracle.reduce([big] * 64)
    assert g[0] == np.float32(64 * 65504.0)
    key = synth.stream_key(0, synth.GRAD, 2, 1, 0)
    h = synth.values_f16(key, 1e-3 * 65536, 0, 4096)
    assert np.all(np.isfinite(oracle.reduce([h] * 8)))
