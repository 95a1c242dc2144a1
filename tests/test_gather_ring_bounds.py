"""CPU check of the gather's aligned-copy kernel: its tile and chunk walk, restated.

The host cuts each layer at shard boundaries into segments and numbers 64 KiB tiles
across them; CTA b of a G-CTA grid takes tiles b, b + G, ... For each tile the first
`head` elements (up to the first 16-byte-aligned destination address) and the elements
after the 16-byte-aligned body are copied one by one by the edge warps; thread 0 streams
the bodies of all of its tiles, cut into chunks of at most 32 KiB, through a ring of S
shared-memory buffers: S - 1 loads are issued ahead, chunk c is stored from buffer c % S
once it has landed, and then the load of chunk c + S - 1 goes into buffer (c - 1) % S.

Checked here, over random layer layouts whose layers start on 8-element boundaries (the
ones the host sends to this kernel): every bulk copy starts on 16-byte boundaries on both
sides and moves a multiple of 16 bytes, at most one buffer's worth; every destination
element is written exactly once, from the right source element; the issuing walk visits
the chunks in the order they are consumed; and a buffer is refilled only after the store
that last read it is no longer the newest one (so waiting for all but the newest store
group to finish reading frees it).
"""
import bisect
import random

import numpy as np
import pytest

TILE = 32768            # elements per tile
CHUNK = 32768           # bytes per ring buffer
SHARD_BASE = 1 << 30    # synthetic byte addresses (16-byte aligned bases)
LAYER_BASE = 1 << 50


def plan_segments(offs, s, nd, shard_addr, layer_addr):
    """The host's cut: (src byte address, dst byte address, elements, first tile)."""
    segs, tiles = [], 0
    for l in range(len(offs) - 1):
        a, b = offs[l], offs[l + 1]
        r = a // s
        while a < b and r < nd and r * s < b:
            lo, hi = max(a, r * s), min(b, (r + 1) * s)
            if hi > lo:
                src = shard_addr[r] + 2 * (lo - r * s)
                dst = layer_addr[l] + 2 * (lo - a)
                assert (src - dst) % 16 == 0  # the aligned class only
                segs.append((src, dst, hi - lo, tiles))
                tiles += -(-(hi - lo) // TILE)
            r += 1
    return segs, tiles


def tile_geom(segs, t):
    seg = bisect.bisect_right([sg[3] for sg in segs], t) - 1
    src, dst, n_seg, first = segs[seg]
    e0 = (t - first) * TILE
    n = min(TILE, n_seg - e0)
    sa, da = src + 2 * e0, dst + 2 * e0
    head = min(((16 - (da & 15)) & 15) >> 1, n)
    body = 0 if (sa + 2 * head) & 15 else ((n - head) >> 3) << 3
    return sa, da, n, head, body


def chunks_of_cta(segs, tiles, b, grid):
    out = []
    for t in range(b, tiles, grid):
        sa, da, n, head, body = tile_geom(segs, t)
        off = 0
        while off < 2 * body:
            ln = min(CHUNK, 2 * body - off)
            out.append((sa + 2 * head + off, da + 2 * head + off, ln))
            off += ln
    return out


def layout(rng):
    nd = rng.choice([1, 2, 3, 8, 64])
    s = 8 * rng.randrange(1, 40000)
    n = rng.randrange(1, nd * s + 1)
    cuts = sorted({0, n} | {8 * rng.randrange(0, n // 8 + 1) for _ in range(rng.randrange(0, 6))})
    return nd, s, cuts


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("stages", [3, 6, 7])
def test_chunk_walk_covers_each_element_once_with_aligned_bulk_copies(seed, stages):
    rng = random.Random(seed * 10 + stages)
    for _ in range(60):
        nd, s, offs = layout(rng)
        shard_addr = [SHARD_BASE + (r << 32) for r in range(nd)]
        layer_addr = [LAYER_BASE + (l << 32) for l in range(len(offs) - 1)]
        segs, tiles = plan_segments(offs, s, nd, shard_addr, layer_addr)
        if tiles == 0:
            continue
        grid = rng.choice([1, 2, 7, 152])
        written = [np.zeros(offs[l + 1] - offs[l], np.int32) for l in range(len(offs) - 1)]

        def put(dst_byte, src_byte, m):
            """m elements from src_byte to dst_byte: inside one layer and one shard, and
            the same flat indices on both sides."""
            l = (dst_byte - LAYER_BASE) >> 32
            r = (src_byte - SHARD_BASE) >> 32
            j = (dst_byte - layer_addr[l]) // 2
            k = (src_byte - shard_addr[r]) // 2
            assert 0 <= j and j + m <= len(written[l]) and 0 <= k and k + m <= s
            assert offs[l] + j == r * s + k
            written[l][j:j + m] += 1

        g = min(grid, tiles)
        for b in range(g):
            ch = chunks_of_cta(segs, tiles, b, g)
            for src, dst, ln in ch:
                assert src % 16 == 0 and dst % 16 == 0 and ln % 16 == 0 and 0 < ln <= CHUNK
                put(dst, src, ln // 2)
            # ring discipline: chunk c lands in buffer c % S; the load of chunk c + S - 1
            # is issued after the store of chunk c, into the buffer last read by the store
            # of chunk c - 1, which by then is not the newest store group
            for c in range(len(ch)):
                nxt = c + stages - 1
                if nxt < len(ch):
                    assert nxt % stages == (c - 1) % stages
                    assert nxt - stages < c  # the buffer's last reader is not chunk c
            # the edge warps: heads and tails of this CTA's tiles
            for t in range(b, tiles, g):
                sa, da, n, head, body = tile_geom(segs, t)
                if head:
                    put(da, sa, head)
                if head + body < n:
                    put(da + 2 * (head + body), sa + 2 * (head + body), n - head - body)
        assert all((x == 1).all() for x in written)
