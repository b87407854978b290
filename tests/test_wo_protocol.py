"""Model of the mbarrier hand-off protocol of the W_O projection kernel
(csrc/pa_wo.cu), run under random schedules on the CPU.

Roles (per CTA): the copy thread (warp 4) fills stage c % S with chunk c (W
tiles and the o box) once the MMAs of chunk c - S are complete; the three
converter warps turn the o box of chunk c into the bf16 hi / lo tile X[c % 2]
once the MMAs of chunk c - 2 (the previous user of X[c % 2]) are complete;
the MMA thread (warp 0) takes chunk c once its stage is full and X[c % 2] is
converted, and commits `done` (the stage may be refilled) and `xfree` (X may
be rewritten).  MMA completion is asynchronous: an engine retires the issued
MMAs in order, and each commit arrives when everything before it has.
Barrier phases follow the hardware's parity rule.  The asserts check the data
flow (no stage or X tile overwritten before its reader is done, nothing read
before it is written); a missing wait deadlocks or fails an assert.
"""
import random

import pytest

from tests.test_verify_protocol import Bar


class Wo:
    def __init__(self, nch, stages=4):
        self.nch, self.S = nch, stages
        self.full = [Bar(1) for _ in range(stages)]
        self.done = [Bar(1) for _ in range(stages)]
        self.xfull = [Bar(96), Bar(96)]
        self.xfree = [Bar(1), Bar(1)]
        self.fin = Bar(1)
        self.stage = [None] * stages      # chunk held by each stage
        self.x = [None, None]             # chunk converted into each X tile
        self.read_stage = set()           # (chunk) whose stage the MMAs finished reading
        self.conv_read = set()            # chunks whose o box was converted
        self.mma_q = []                   # issued MMAs / commits, retired in order
        self.log = set()

    @staticmethod
    def wait(bar, parity):
        while not bar.ready(parity):
            yield (bar, parity)

    def copier(self):
        for c in range(self.nch):
            if c >= self.S:
                pc = c - self.S
                yield from self.wait(self.done[pc % self.S], (pc // self.S) & 1)
                assert pc in self.read_stage and pc in self.conv_read, "stage refilled while read"
            self.stage[c % self.S] = c
            self.full[c % self.S].arrive()    # the copy lands (expect_tx + bytes)

    def converter(self):
        for c in range(self.nch):
            st = c % self.S
            yield from self.wait(self.full[st], (c // self.S) & 1)
            assert self.stage[st] == c, "o box read before its copy landed"
            if c >= 2:
                yield from self.wait(self.xfree[c & 1], ((c >> 1) - 1) & 1)
                assert ("mma_done", c - 2) in self.log, "X rewritten while the MMAs read it"
            self.x[c & 1] = c
            self.conv_read.add(c)
            self.xfull[c & 1].arrive(96)

    def mma(self):
        for c in range(self.nch):
            st = c % self.S
            yield from self.wait(self.full[st], (c // self.S) & 1)
            yield from self.wait(self.xfull[c & 1], (c >> 1) & 1)
            assert self.stage[st] == c and self.x[c & 1] == c, "MMA before its operands"
            self.mma_q.append(("mma", c))
            self.mma_q.append(("commit", self.done[st]))
            self.mma_q.append(("commit", self.xfree[c & 1]))
        self.mma_q.append(("commit", self.fin))
        yield from self.wait(self.fin, 0)

    def engine(self):
        while True:
            if self.mma_q:
                kind, v = self.mma_q.pop(0)
                if kind == "mma":
                    # the operands must still hold chunk v while the MMA runs
                    assert self.stage[v % self.S] == v and self.x[v & 1] == v, "operand overwritten"
                    self.read_stage.add(v)
                    self.log.add(("mma_done", v))
                else:
                    v.arrive()
            yield None

    def run(self, seed):
        rng = random.Random(seed)
        roles = {"copy": self.copier(), "conv": self.converter(), "mma": self.mma()}
        eng = self.engine()
        blocked = {a: None for a in roles}
        alive = set(roles)
        idle = 0
        while alive:
            progress = False
            order = sorted(alive)
            rng.shuffle(order)
            for a in order[: rng.randint(1, len(order))]:
                w = blocked[a]
                if w is not None and not w[0].ready(w[1]):
                    continue
                try:
                    blocked[a] = next(roles[a])
                except StopIteration:
                    alive.discard(a)
                progress = True
            if rng.random() < 0.5:
                next(eng)
            if not progress and not self.mma_q:
                idle += 1
                if idle > 3:
                    raise AssertionError(f"deadlock: {sorted(alive)}")
            else:
                idle = 0
        assert not self.mma_q


@pytest.mark.parametrize("nch", [1, 2, 3, 4, 5, 7, 14, 15])
def test_wo_protocol_random_schedules(nch):
    for seed in range(30):
        Wo(nch).run(seed)


def test_model_catches_a_missing_xfree_wait():
    """A converter that rewrites X without waiting for the MMAs two chunks
    back is caught (under some schedules)."""
    class Broken(Wo):
        def converter(self):
            for c in range(self.nch):
                st = c % self.S
                yield from self.wait(self.full[st], (c // self.S) & 1)
                self.x[c & 1] = c
                self.conv_read.add(c)
                self.xfull[c & 1].arrive(96)

    with pytest.raises(AssertionError):
        for seed in range(80):
            Broken(14).run(seed)


def test_model_catches_an_early_refill():
    """A copy thread that refills a stage without waiting for its MMAs is
    caught."""
    class Broken(Wo):
        def copier(self):
            for c in range(self.nch):
                self.stage[c % self.S] = c
                self.full[c % self.S].arrive()
                yield None

    with pytest.raises(AssertionError):
        for seed in range(80):
            Broken(14).run(seed)
