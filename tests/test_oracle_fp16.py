"""Pins of the oracle's fp16 conversions against numpy's IEEE binary16 conversions.

fp16 <-> fp32 is exhaustive in both directions: all 65536 fp16 patterns against numpy,
and all 2^32 fp32 patterns against torch's conversion (chunks of 2^24 on all host
threads). The structured cases below (every sign, exponent and top-10 fraction bits with
the rounding-critical low-bit patterns; the fp16 subnormal range; the overflow threshold)
are also checked against numpy, a second independent conversion.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle


def f16_bits_numpy(x):
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def same_f16(a, b):
    """Bitwise equality, with any NaN equal to any NaN."""
    a = np.asarray(a, dtype=np.uint16)
    b = np.asarray(b, dtype=np.uint16)
    a_nan = ((a & 0x7C00) == 0x7C00) & ((a & 0x03FF) != 0)
    b_nan = ((b & 0x7C00) == 0x7C00) & ((b & 0x03FF) != 0)
    return np.all(np.where(a_nan | b_nan, a_nan == b_nan, a == b))


def test_f16_to_f32_exhaustive():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_structured():
    hi = np.arange(1 << 19, dtype=np.uint32) << np.uint32(13)  # sign, exponent, top 10
    lows = np.array([0, 1, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x0800, 0x1800], dtype=np.uint32)
    bits = (hi[:, None] | lows[None, :]).ravel()
    x = bits.view(np.float32)
    assert same_f16(oracle.f32_to_f16(x), f16_bits_numpy(x))


def test_f32_to_f16_subnormal_and_overflow_ranges():
    # fp32 exponents 2^-26 .. 2^-14 (inputs whose fp16 result is subnormal, zero or the
    # smallest normal), every fraction, positive sign; then the overflow edge
    for e in range(127 - 26, 127 - 13):
        bits = (np.uint32(e) << np.uint32(23)) | np.arange(1 << 23, dtype=np.uint32)
        x = bits.view(np.float32)
        assert same_f16(oracle.f32_to_f16(x), f16_bits_numpy(x)), e
        assert same_f16(oracle.f32_to_f16(-x), f16_bits_numpy(-x)), e
    edge = np.float32(65520.0).view(np.uint32)
    bits = np.arange(edge - 4096, edge + 4096, dtype=np.uint32)
    x = bits.view(np.float32)
    assert same_f16(oracle.f32_to_f16(x), f16_bits_numpy(x))
    assert oracle.f32_to_f16(np.array([65519.996], dtype=np.float32))[0] == 0x7BFF
    assert oracle.f32_to_f16(np.array([65520.0], dtype=np.float32))[0] == 0x7C00


def test_f32_to_f16_exhaustive():
    def chunk(k):
        bits = np.arange(1 << 24, dtype=np.uint32) + np.uint32(k << 24)
        x = bits.view(np.float32)
        ref = torch.from_numpy(x).half().view(torch.int16).numpy().view(np.uint16)
        return k if not same_f16(oracle.f32_to_f16(x), ref) else None

    with ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
        bad = [k for k in ex.map(chunk, range(256)) if k is not None]
    assert bad == []


def test_f32_to_f16_special_values():
    x = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1.0, -2.0, 65504.0, 2.0**-24,
                  2.0**-25, 3 * 2.0**-26, 2.0**-14], dtype=np.float32)
    got = oracle.f32_to_f16(x)
    assert list(got[:4]) == [0x0000, 0x8000, 0x7C00, 0xFC00]
    assert (got[4] & 0x7C00) == 0x7C00 and (got[4] & 0x3FF) != 0
    assert list(got[5:]) == [0x3C00, 0xC000, 0x7BFF, 0x0001, 0x0000, 0x0001, 0x0400]

