"""Pins of the oracle's ZeRO-3 parameter gather against slicing and brute force.

The all-gather before forward (ZeRO explainer, Chapter 02, ZeRO-3 item) reassembles the
fp16 shards; layer l is a contiguous slice of the flat buffer they concatenate to.
"""
import numpy as np

import oracle


def make_shards(rng, nd, s):
    return [rng.integers(0, 65536, s, dtype=np.uint64).astype(np.uint16) for _ in range(nd)]


def test_gather_equals_slices_of_concatenation():
    rng = np.random.default_rng(20)
    for nd, s, offs in [
        (1, 16, [0, 16]),
        (4, 8, [0, 5, 9, 20, 32]),            # odd offsets, a layer spanning three shards
        (3, 24, [0, 1, 2, 70]),               # one-element layers
        (8, 16, [0, 0, 64, 64, 100]),         # empty layers
        (64, 40, [l * 64 for l in range(41)]),  # 40 equal layers over 64 shards
    ]:
        shards = make_shards(rng, nd, s)
        flat = np.concatenate(shards)
        out = oracle.gather(shards, s, offs)
        assert len(out) == len(offs) - 1
        for l, d in enumerate(out):
            assert np.array_equal(d, flat[offs[l]:offs[l + 1]])


def test_gather_source_brute_force():
    for s in [1, 7, 8, 203]:
        nd = 5
        owner = np.repeat(np.arange(nd), s)
        local = np.tile(np.arange(s), nd)
        for i in range(nd * s):
            assert oracle.gather_source(s, i) == (owner[i], local[i])
