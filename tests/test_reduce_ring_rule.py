"""CPU check of the bulk-load reduce's tile claiming and stage ring, restated.

In each CTA a producer thread claims tiles of TG groups (groups of 8 elements) from a
shared counter when it needs the next one and, for each tile, takes the ranks RC at a time
(RC = min(Nd, 2048 / consumers): 8 with 256 consumers, 4 with 512; a rank count known only
at run time uses the full RC with a shorter last chunk). Each chunk is one
stage of an S-stage ring: the producer waits until the stage's previous contents have
been consumed, records (tile, chunk) in it and bulk-loads the chunk's ranks, rank-major,
nv * 16 bytes each (nv = the tile's groups). Consumer thread c owns groups c + 256 j of
each tile and adds the chunk's ranks in order; after the tile's last chunk it writes the
group's sums. An end mark closes the stream.

Here the producers and consumers of a grid of CTAs run with their actions interleaved at
random. Checked: every stage holds at most 32 KiB and each rank's slice lies inside the
stage; a stage is refilled only after every consumer is done with it; every group of the
span gets the ranks 0..Nd-1 added exactly once each, in rank order, and its sums written
exactly once; and every CTA ends on the end mark.
"""
import random

import pytest

STAGE_BYTES = 32768


def geometry(nd, nd_static, consumers):
    ranks = 2048 // consumers  # ranks per 32 KiB stage, one group per consumer
    rc = nd_static if 0 < nd_static < ranks else ranks
    g = 1 if rc >= ranks else ranks // rc
    return rc, g, consumers * g


class Cta:
    def __init__(self, nd, nd_static, n_vec, stages, counter, log, consumers):
        self.nd, self.n_vec, self.S, self.consumers = nd, n_vec, stages, consumers
        self.rc, self.g, self.tg = geometry(nd, nd_static, consumers)
        self.tiles = -(-n_vec // self.tg)
        self.nchunks = -(-nd // self.rc)
        self.counter, self.log = counter, log
        self.stage = [None] * stages      # (tile, chunk) or ('end',)
        self.full = [0] * stages          # phases completed
        self.empty = [0] * stages
        self.q_prod = self.q_cons = 0
        self.pending = []                 # (tile, chunk) the producer still has to issue
        self.prod_done = False
        self.next_claim = None
        self.cons_done = False

    def claim(self):
        t = self.counter[0]
        self.counter[0] += 1
        return t

    def produce(self):
        """One producer action; False if it has to wait."""
        if self.prod_done:
            return False
        s = self.q_prod % self.S
        if self.q_prod >= self.S and self.empty[s] < self.q_prod // self.S:
            return False  # the stage's previous contents are not consumed yet
        if not self.pending:
            t = self.claim()
            if t >= self.tiles:
                self.stage[s] = ('end',)
                self.full[s] += 1
                self.q_prod += 1
                self.prod_done = True
                return True
            self.pending = [(t, k) for k in range(self.nchunks)]
        t, k = self.pending.pop(0)
        v0 = t * self.tg
        nv = min(self.tg, self.n_vec - v0)
        nr = min(self.rc, self.nd - k * self.rc)
        for j in range(nr):  # rank-major slices, each inside the stage
            lo, hi = j * self.tg * 16, j * self.tg * 16 + nv * 16
            assert 0 <= lo and hi <= STAGE_BYTES
        self.stage[s] = (t, k)
        self.full[s] += 1
        self.q_prod += 1
        return True

    def consume(self):
        """All consumers take the next stage together (each reads its own groups)."""
        if self.cons_done:
            return False
        s = self.q_cons % self.S
        if self.full[s] <= self.q_cons // self.S:
            return False  # not landed yet
        ent = self.stage[s]
        if ent == ('end',):
            self.cons_done = True
            return True
        t, k = ent
        v0 = t * self.tg
        nv = min(self.tg, self.n_vec - v0)
        nr = min(self.rc, self.nd - k * self.rc)
        for c in range(self.consumers):
            for j in range(self.g):
                gi = c + self.consumers * j
                if gi >= nv:
                    continue
                v = v0 + gi
                self.log.setdefault(v, []).extend(k * self.rc + r for r in range(nr))
                if k == self.nchunks - 1:
                    self.log.setdefault(('written', v), 0)
                    self.log[('written', v)] += 1
        self.empty[s] += 1
        self.q_cons += 1
        return True


# the rank counts the library sends to this kernel: 8, 16, 32 and 64 with the count fixed
# at compile time, the others read at run time
@pytest.mark.parametrize("nd,nd_static", [(8, 8), (16, 16), (32, 32), (64, 64), (9, 0), (17, 0),
                                          (100, 0), (256, 0)])
@pytest.mark.parametrize("stages", [3, 6])
@pytest.mark.parametrize("consumers", [256, 512])
def test_every_group_sums_all_ranks_once_in_order(nd, nd_static, stages, consumers):
    rng = random.Random(nd * 7 + stages + consumers)
    for n_vec in [1, 255, 256, 257, 1000, 5000, rng.randrange(1, 20000)]:
        counter, log = [0], {}
        rc, g, tg = geometry(nd, nd_static, consumers)
        tiles = -(-n_vec // tg)
        grid = min(rng.choice([1, 2, 5, 152]), tiles)
        ctas = [Cta(nd, nd_static, n_vec, stages, counter, log, consumers) for _ in range(grid)]
        live = list(ctas)
        while live:
            c = rng.choice(live)
            moved = c.produce() if rng.random() < 0.5 else c.consume()
            if not moved:
                moved = c.consume() or c.produce()
            if c.cons_done and c.prod_done:
                live.remove(c)
            else:
                assert moved or any(x is not c for x in live) or c.produce() or c.consume()
        for v in range(n_vec):
            assert log[v] == list(range(nd)), v
            assert log[('written', v)] == 1
        assert counter[0] == tiles + grid  # every CTA's last claim fell past the end
