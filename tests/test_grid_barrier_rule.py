"""CPU check of the one-launch step's grid barrier rule, restated.

The barrier keeps one 64-bit arrival count that only grows. A CTA adds 1 and gets the
count before its arrival, `old`; its launch's barrier is complete when the count reaches
target = old - old % n + n (n CTAs per launch), and the CTA that makes old + 1 == target
is the last to arrive. Launches that use the count follow one another (stream order), so
launch k's arrivals take it from k*n to (k+1)*n. Here, over many launches with random
arrival orders: every CTA of a launch computes the same target, exactly one CTA is the
last, and no CTA could see the count at its target before the last arrival of its own
launch (a waiter's condition count >= target only becomes true then).
"""
import random

import pytest


@pytest.mark.parametrize("n", [1, 2, 3, 152, 160])
def test_every_cta_of_a_launch_waits_for_exactly_its_launch(n):
    rng = random.Random(n)
    count = 0
    for k in range(40):
        order = list(range(n))
        rng.shuffle(order)
        targets, lasts = set(), 0
        for pos, _ in enumerate(order):
            old = count
            count += 1
            target = old - old % n + n
            targets.add(target)
            lasts += old + 1 == target
            # before the launch's last arrival the count is below every waiter's target
            if pos < n - 1:
                assert count < target
        assert targets == {(k + 1) * n} and lasts == 1 and count == (k + 1) * n
