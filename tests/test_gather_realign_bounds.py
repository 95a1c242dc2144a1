"""CPU check of the gather's realigning path: its index arithmetic, restated, over many
source/destination offsets and tile lengths.

For a tile of n fp16 elements whose source and destination differ in alignment modulo 16
bytes, the kernel stores aligned 16-byte destination vectors j in [j_lo, j_hi), each built
from the aligned source blocks W_j and W_{j+1}, and copies the remaining elements one by
one. Here every load must lie inside the tile's source bytes, and every destination element
must be written exactly once, from the right source element.
"""
import random

import pytest


def plan(sa, da, n):
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


@pytest.mark.parametrize("seed", range(4))
def test_realign_reads_stay_inside_and_cover_each_element_once(seed):
    rng = random.Random(seed)
    checked = 0
    for _ in range(5000):
        sa = 4096 + 2 * rng.randrange(64)
        da = 8192 + 2 * rng.randrange(64)
        n = rng.choice([rng.randrange(1, 40), rng.randrange(1, 3000), 32768])
        if (sa - da) % 16 == 0:
            continue
        head, d, a, j_lo, j_hi, v0, v1 = plan(sa, da, n)
        written = [0] * n
        for j in range(j_lo, j_hi):
            for blk in (a + 16 * j, a + 16 * (j + 1)):
                assert sa <= blk and blk + 16 <= sa + 2 * n
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
