"""CPU check of the one-launch step's counting sums (its grid barrier), restated.

Each of W words takes one atomic add per CTA of `2^48 + v` (v < 2^32): bits 48..63 count
the CTAs that have added, bits 0..47 hold the sum of their values. A waiting warp accepts
the words once every count equals the grid size n, and takes the sums from the same
reads. Launch k (the launch count read by every CTA at its start) uses word set k & 1;
its CTA 0 clears set (k + 1) & 1 at its start and stores k + 1 into the count after its
own wait, whether or not the wait completed.

Here, with the adds, reads and clears of many launches interleaved at random (each word
only ever sees whole atomic adds, in some order): a read with every count complete holds
the exact sums of that launch's values; no read of an incomplete set is accepted; a
launch in which a CTA never adds ends with its waits given up, and the launches after it
are exact again; the four 32-bit limbs put back together give the 128-bit sum of the
CTAs' 128-bit partials.
"""
import random

import pytest

SHIFT = 48
ONE = 1 << SHIFT
W = 5
MASK128 = (1 << 128) - 1


def limbs(x128, bad):
    return [x128 & 0xFFFFFFFF, (x128 >> 32) & 0xFFFFFFFF, (x128 >> 64) & 0xFFFFFFFF,
            (x128 >> 96) & 0xFFFFFFFF, bad]


def assemble(l0, l1, l2, l3):
    """The kernel's reassembly: l0 + l1 2^32 + l2 2^64 + l3 2^96, modulo 2^128."""
    return (l0 + (l1 << 32) + (l2 << 64) + (l3 << 96)) & MASK128


def run_launch(rng, sets, k, n, skip=None, polls=50):
    """One launch; returns the sums each CTA accepted (None where its wait gave up)."""
    partials = [(rng.getrandbits(rng.choice([1, 40, 100, 107])), rng.randrange(0, 30000))
                for _ in range(n)]
    words = sets[k & 1]
    # CTA 0 clears the next launch's set at its start
    for j in range(W):
        sets[(k + 1) & 1][j] = 0
    adds = [(c, j) for c in range(n) if c != skip for j in range(W)]
    rng.shuffle(adds)
    accepted = [None] * n
    polls_left = [polls] * n
    waiting = [c for c in range(n) if c != skip]
    while adds or waiting:
        if adds and rng.random() < 0.6:
            c, j = adds.pop()
            v = limbs(*partials[c])[j]
            assert v < 2 ** 32 or j == 4
            words[j] = (words[j] + ONE + v) % (1 << 64)
            continue
        if not waiting:
            continue
        c = rng.choice(waiting)
        read = list(words)  # one read per lane, one after another
        if all(w >> SHIFT == n for w in read):
            accepted[c] = [w & (ONE - 1) for w in read]
            waiting.remove(c)
        else:
            polls_left[c] -= 1
            if polls_left[c] == 0 and not adds:
                waiting.remove(c)  # gave up
    want = [sum(limbs(*partials[c])[j] for c in range(n) if c != skip) for j in range(W)]
    ss = sum(partials[c][0] for c in range(n) if c != skip) & MASK128
    bad = sum(partials[c][1] for c in range(n) if c != skip)
    return accepted, want, ss, bad


@pytest.mark.parametrize("n", [1, 2, 3, 152, 160])
def test_counting_sums_are_exact_and_complete_only_with_every_cta(n):
    rng = random.Random(n)
    sets = [[0] * W, [0] * W]
    k = 0
    for launch in range(12):
        skip = rng.randrange(n) if launch in (4, 5) and n > 1 else None
        accepted, want, ss, bad = run_launch(rng, sets, k, n, skip)
        if skip is None:
            for a in accepted:
                assert a == want
                assert assemble(*a[:4]) == ss and a[4] == bad
        else:
            assert all(a is None for a in accepted)  # nobody accepts an incomplete set
        k += 1  # CTA 0 stores k + 1 after its wait in either case


def test_the_count_never_takes_a_carry_from_the_sum():
    # the largest values from the most CTAs the field allows
    n = (1 << 16) - 1
    w = sum(ONE + (2 ** 32 - 1) for _ in range(n))
    assert w >> SHIFT == n and w & (ONE - 1) == n * (2 ** 32 - 1)
    assert w < 1 << 64
