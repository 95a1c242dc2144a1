"""CPU check of the gather's aligned-copy kernel: its tile claiming and ring, restated.

The host cuts each layer at shard boundaries into segments and numbers fixed-size tiles
across them (32 KiB, the kernel's; 64 KiB is checked too). In each CTA of the launch,
thread 0 claims tiles from a shared counter (an atomic add, one when it needs one), queues
the ones with a 16-byte-aligned body, and streams the bodies, cut
into chunks of at most 32 KiB, through a ring of S shared-memory buffers: it keeps S - 1
loads in flight, stores chunk c from buffer c % S once it has landed, and issues the next
load into a buffer only after waiting for every store but the newest to finish reading.
The other warps copy every tile's unaligned edge elements, the tiles split statically
over the CTAs. The last CTA to finish resets the counter.

Here that state machine runs for every CTA of a grid, the CTAs' actions interleaved at
random (so the claims land in arbitrary order), over random layer layouts whose layers
start on 8-element boundaries (the ones the host sends to this kernel). Checked: every
bulk copy starts on 16-byte boundaries on both sides and moves a positive multiple of
16 bytes, at most one buffer's worth; each store sends out the bytes its buffer's last
load brought in, for the same element; a buffer is refilled only when the store that last
read it is not the newest one; the claim queue never overflows; every destination
element is written exactly once, from the right source element; and every CTA stops
claiming only once the counter has passed the last tile.
"""
import bisect
import random

import numpy as np
import pytest

TILES = (16384, 32768)  # elements per tile (the kernel's 32 KiB, and 64 KiB)
CHUNK = 32768           # bytes per ring buffer
SHARD_BASE = 1 << 30    # synthetic byte addresses (16-byte aligned bases)
LAYER_BASE = 1 << 50


def plan_segments(offs, s, nd, shard_addr, layer_addr, tile):
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
                tiles += -(-(hi - lo) // tile)
            r += 1
    return segs, tiles


def tile_geom(segs, t, tile):
    seg = bisect.bisect_right([sg[3] for sg in segs], t) - 1
    src, dst, n_seg, first = segs[seg]
    e0 = (t - first) * tile
    n = min(tile, n_seg - e0)
    sa, da = src + 2 * e0, dst + 2 * e0
    head = min(((16 - (da & 15)) & 15) >> 1, n)
    body = 0 if (sa + 2 * head) & 15 else ((n - head) >> 3) << 3
    return sa, da, n, head, body


class Cta:
    """Thread 0 of one CTA: claim queue, producer (loads) and consumer (stores)."""

    def __init__(self, stages, queue, segs, tiles, counter, copy, tile):
        self.S, self.Q, self.tile = stages, queue, tile
        self.segs, self.tiles, self.counter, self.copy = segs, tiles, counter, copy
        self.q = [None] * queue
        self.q_head = self.q_tail = 0
        self.p_idx = self.p_off = self.c_off = 0
        self.claims_done = False
        self.issued = self.done = 0
        self.buf = [None] * stages       # (src, len) of each buffer's last load
        self.reader = [None] * stages    # chunk index of each buffer's last store
        self.last_claim = -1

    def claim(self):
        while not self.claims_done and self.q_tail - self.q_head < self.Q:
            t = self.counter[0]
            self.counter[0] += 1
            if t >= self.tiles:
                self.claims_done = True
                break
            assert t > self.last_claim  # a CTA's claims increase (its segment index runs)
            self.last_claim = t
            sa, da, n, head, body = tile_geom(self.segs, t, self.tile)
            if body == 0:
                continue
            self.q[self.q_tail % self.Q] = (sa + 2 * head, da + 2 * head, 2 * body)
            self.q_tail += 1
            return True
        assert self.q_tail - self.q_head < self.Q or self.claims_done
        return False

    def fill(self):
        while self.issued - self.done < self.S - 1:
            if self.p_idx == self.q_tail and not self.claim():
                return
            src, dst, nbytes = self.q[self.p_idx % self.Q]
            ln = min(CHUNK, nbytes - self.p_off)
            s = self.issued % self.S
            # wait for every store but the newest to finish reading: this buffer's last
            # reader must be older than the newest store (chunk done - 1)
            if self.reader[s] is not None:
                assert self.reader[s] <= self.done - 2
            assert (src + self.p_off) % 16 == 0 and ln % 16 == 0 and 0 < ln <= CHUNK
            self.buf[s] = (src + self.p_off, ln)
            self.issued += 1
            self.p_off += ln
            if self.p_off == nbytes:
                self.p_idx += 1
                self.p_off = 0

    def consume(self):
        """One iteration of the main loop; False once the CTA is done."""
        if self.done == self.issued:
            return False
        src, dst, nbytes = self.q[self.q_head % self.Q]
        ln = min(CHUNK, nbytes - self.c_off)
        s = self.done % self.S
        b_src, b_len = self.buf[s]
        assert b_len == ln and b_src == src + self.c_off
        assert (dst + self.c_off) % 16 == 0
        self.copy(dst + self.c_off, b_src, ln // 2)
        self.reader[s] = self.done
        self.done += 1
        self.c_off += ln
        if self.c_off == nbytes:
            self.q_head += 1
            self.c_off = 0
        self.fill()
        return True


def layout(rng):
    nd = rng.choice([1, 2, 3, 8, 64])
    s = 8 * rng.randrange(1, 40000)
    n = rng.randrange(1, nd * s + 1)
    cuts = sorted({0, n} | {8 * rng.randrange(0, n // 8 + 1) for _ in range(rng.randrange(0, 6))})
    return nd, s, cuts


@pytest.mark.parametrize("seed", range(2))
@pytest.mark.parametrize("stages", [3, 4, 6, 7])
@pytest.mark.parametrize("tile", TILES)
def test_claims_and_ring_cover_each_element_once(seed, stages, tile):
    rng = random.Random(seed * 10 + stages + tile)
    for _ in range(40):
        nd, s, offs = layout(rng)
        shard_addr = [SHARD_BASE + (r << 32) for r in range(nd)]
        layer_addr = [LAYER_BASE + (l << 32) for l in range(len(offs) - 1)]
        segs, tiles = plan_segments(offs, s, nd, shard_addr, layer_addr, tile)
        if tiles == 0:
            continue
        grid = min(rng.choice([1, 2, 7, 152]), tiles)
        written = [np.zeros(offs[l + 1] - offs[l], np.int32) for l in range(len(offs) - 1)]

        def copy(dst_byte, src_byte, m):
            """m elements from src_byte to dst_byte: inside one layer and one shard, and
            the same flat indices on both sides."""
            l = (dst_byte - LAYER_BASE) >> 32
            r = (src_byte - SHARD_BASE) >> 32
            j = (dst_byte - layer_addr[l]) // 2
            k = (src_byte - shard_addr[r]) // 2
            assert 0 <= j and j + m <= len(written[l]) and 0 <= k and k + m <= s
            assert offs[l] + j == r * s + k
            written[l][j:j + m] += 1

        counter = [0]
        ctas = [Cta(stages, stages + 2, segs, tiles, counter, copy, tile) for _ in range(grid)]
        for c in ctas:
            c.fill()
        live = list(ctas)
        while live:
            c = rng.choice(live)
            if not c.consume():
                live.remove(c)
        # every CTA made its last claim past the end before it stopped, so the counter
        # holds one failed claim per CTA when the last one resets it
        assert all(c.claims_done for c in ctas) and counter[0] == tiles + grid
        # the edge warps: heads and tails of every tile, split statically over the CTAs
        for b in range(grid):
            for t in range(b, tiles, grid):
                sa, da, n, head, body = tile_geom(segs, t, tile)
                if body == 0:
                    copy(da, sa, n)
                    continue
                if head:
                    copy(da, sa, head)
                if head + body < n:
                    copy(da + 2 * (head + body), sa + 2 * (head + body), n - head - body)
        assert all((x == 1).all() for x in written)
