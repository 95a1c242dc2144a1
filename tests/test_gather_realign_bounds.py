"""CPU check of the gather's realigning path: its index arithmetic, restated, over many
source/destination offsets and tile lengths.

For a tile of n fp16 elements whose source and destination differ in alignment modulo 16
bytes, the kernel stores aligned 16-byte destination vectors j in [j_lo, j_hi), each built
from the aligned source blocks W_j and W_{j+1}, and copies the elements outside [v0, v1)
one by one. The vectors are cut into stretches of up to 2048; one bulk load brings a
stretch's blocks W_jb .. W_{jb+nv} into a ring stage of 32896 bytes. Here every load must
lie inside the tile's source bytes and fit its stage, every destination element must be
written exactly once from the right source element, and the order in which thread 0
issues stretches must be the order in which the CTA consumes them.
"""
import random

import pytest

STRETCH = 2048
STAGE_BYTES = 32768 + 128
TILE = 32768


def geometry(sa, da, n):
    head = min(((16 - (da & 15)) & 15) >> 1, n)
    s_body = sa + 2 * head
    d = s_body & 15
    a = s_body - d
    s_end = sa + 2 * n
    nvec = (n - head) >> 3
    j_lo = 0 if a >= sa else 1
    j_hi = ((s_end - a - 16) >> 4) if s_end >= a + 16 else 0
    j_hi = max(min(j_hi, nvec), j_lo)
    v0, v1 = min(head + 8 * j_lo, n), min(head + 8 * j_hi, n)
    return head, d, a, j_lo, j_hi, v0, v1


def stretches(j_lo, j_hi):
    return [(jb, min(STRETCH, j_hi - jb)) for jb in range(j_lo, j_hi, STRETCH)]


@pytest.mark.parametrize("seed", range(4))
def test_realign_reads_stay_inside_and_cover_each_element_once(seed):
    rng = random.Random(seed)
    checked = 0
    for _ in range(5000):
        sa = 4096 + 2 * rng.randrange(64)
        da = 8192 + 2 * rng.randrange(64)
        n = rng.choice([rng.randrange(1, 40), rng.randrange(1, 3000), rng.randrange(1, TILE + 1),
                        TILE])
        if (sa - da) % 16 == 0:
            continue
        head, d, a, j_lo, j_hi, v0, v1 = geometry(sa, da, n)
        assert d in range(2, 16, 2) or (head == n and j_lo == j_hi)
        written = [0] * n
        for jb, nv in stretches(j_lo, j_hi):
            load0, nbytes = a + 16 * jb, 16 * (nv + 1)
            assert load0 % 16 == 0 and nbytes <= STAGE_BYTES
            assert sa <= load0 and load0 + nbytes <= sa + 2 * n
            for i in range(nv):
                j = jb + i
                assert 16 * (i + 1) + 16 <= nbytes  # W_{j+1} is in the stage
                for e in range(8):
                    di = head + 8 * j + e
                    assert 0 <= di < n
                    assert (a + 16 * j + d + 2 * e - sa) // 2 == di  # source element == dest
                    written[di] += 1
        for i in list(range(v0)) + list(range(v1, n)):
            written[i] += 1
        assert written == [1] * n
        assert head == n or (da + 2 * head) % 16 == 0
        checked += 1
    assert checked > 3000


def test_issue_order_matches_consumption_order():
    rng = random.Random(7)
    for _ in range(200):
        # one CTA's tiles, each with its vector range; some tiles have no vectors at all
        tiles = []
        for _ in range(rng.randrange(1, 12)):
            j_lo = rng.randrange(2)
            tiles.append((j_lo, max(j_lo, rng.choice([0, 1, 5, 2047, 2048, 2049, 4095, 4096]))))
        consumed = [(t, jb) for t, (lo, hi) in enumerate(tiles) for jb in range(lo, hi, STRETCH)]
        issued, t, h = [], 0, 0  # the issuing walk: tile t, next stretch h of it
        while t < len(tiles):
            lo, hi = tiles[t]
            jb = lo + h * STRETCH
            if jb < hi:
                issued.append((t, jb))
                h += 1
            else:
                t, h = t + 1, 0
        assert issued == consumed
