"""Model of the abort-and-drain exit of the tcgen05 verify kernel
(csrc/pa_verify_umma.cuh), run under random schedules on the CPU.

Every wait of the kernel is capped.  When one runs out, that role sets the
CTA's abort flag and the error bit; every other role's wait returns as soon
as it sees the flag, each role leaves its loops, and before the CTA exits
(tensor memory is released, shared memory handed to the next CTA):
  * each producer lane waits for the last fill it issued into each of its
    stages (a TMA copy still in flight would write into memory the CTA no
    longer owns);
  * the two MMA-issuing threads commit to a common barrier and wait for it,
    so that no tensor-core operation still reads or writes tensor memory.
Copies and MMA completions are asynchronous here: a DMA agent lands issued
copies in random order and one agent per issuing thread retires its MMAs in
order (commit arrivals with them).  A role's n-th wait on a pending barrier
is made to run out; the run must end with every role returned, no copy in
flight and no MMA pending, and without deadlock.  Barrier phases follow the
hardware rule (a wait for parity P passes once the phase of parity P has
completed), so a drain that waits on the wrong phase either passes while a
copy is in flight or never passes; both fail.  A planted mistake -- the
producer counting a fill before its stage is free -- is caught.
"""
import random

import pytest

from tests.test_verify_protocol import TB, Bar, tiles


class Abort(Exception):
    pass


class AbortKernel:
    def __init__(self, items, nrk, nrv, expire=None, count_before_wait=False):
        self.items, self.nrk, self.nrv = items, nrk, nrv
        self.expire = expire                      # (role, n): its n-th pending wait runs out
        self.count_before_wait = count_before_wait
        self.rkfull = [Bar(1) for _ in range(TB * nrk)]
        self.rkfree = [Bar(16) for _ in range(TB * nrk)]
        self.rvfull = [Bar(1) for _ in range(TB * nrv)]
        self.rvfree = [Bar(32) for _ in range(TB * nrv)]
        self.vfull, self.vfree = [Bar(128), Bar(128)], [Bar(1), Bar(1)]
        self.kfull, self.kfree = [Bar(128), Bar(128)], [Bar(1), Bar(1)]
        self.sfull, self.sfree = [Bar(1), Bar(1)], [Bar(256), Bar(256)]
        self.pfull, self.pdone = [Bar(256), Bar(256)], [Bar(1), Bar(1)]
        self.odone, self.ofree, self.done = Bar(1), Bar(256), Bar(2)
        self.abort = False
        self.err = False
        self.pending_waits = {}
        self.inflight = []                        # (lane, barrier) of issued copies
        self.mma = {"qk": [], "pv": []}   # per issuing thread: commits in order

    # -- waits
    def wait_bar(self, bar, parity, who):
        """Capped wait that gives up once another role gave up (wait_bar)."""
        if bar.ready(parity):
            return True
        n = self.pending_waits.get(who, 0)
        self.pending_waits[who] = n + 1
        if self.expire == (who, n):
            self.abort = True
            self.err = True
            return False
        while True:
            yield lambda: bar.ready(parity) or self.abort
            if bar.ready(parity):
                return True
            if self.abort:
                return False

    def drain_wait(self, bar, parity):
        """Capped wait without the abort check."""
        while not bar.ready(parity):
            yield lambda: bar.ready(parity)

    def items_tiles(self, skip_empty=True):
        g = 0
        for n in self.items:
            if n == 0 and skip_empty:
                continue
            tl = tiles(n)
            yield [(g + i, i, len(tl), nb) for i, nb in enumerate(tl)]
            g += len(tl)

    # -- roles
    def producer(self, side, j):
        nr = self.nrk if side == "K" else self.nrv
        full = self.rkfull if side == "K" else self.rvfull
        free = self.rkfree if side == "K" else self.rvfree
        who = f"prod{side}{j}"
        ruse = [0] * nr
        ok = True
        for tl in self.items_tiles(skip_empty=False):
            for g, _, _, nb in tl:
                if j >= nb:
                    continue
                st = g % nr
                use = ruse[st]
                if self.count_before_wait:
                    ruse[st] += 1
                ok = yield from self.wait_bar(free[st * TB + j], (use & 1) ^ 1, who)
                if not ok:
                    break
                if not self.count_before_wait:
                    ruse[st] += 1
                self.inflight.append((who, full[st * TB + j]))   # the copy lands later
            if not ok:
                break
        for a in range(nr):   # the last fill of each stage may still be in flight
            if ruse[a] > 0:
                yield from self.drain_wait(full[a * TB + j], (ruse[a] - 1) & 1)
        assert not any(w == who for w, _ in self.inflight), f"{who}: copy in flight at exit"

    def qk(self):
        ok = True
        for tl in self.items_tiles():
            for g, _, _, _ in tl:
                ok = (yield from self.wait_bar(self.kfull[g & 1], (g >> 1) & 1, "qk")) and \
                     (yield from self.wait_bar(self.sfree[g & 1], ((g >> 1) & 1) ^ 1, "qk"))
                if not ok:
                    break
                self.mma["qk"] += [self.sfull[g & 1], self.kfree[g & 1]]
            if not ok:
                break
        self.mma["qk"].append(self.done)
        yield from self.drain_wait(self.done, 0)

    def pv(self):
        who, ok, oi = "pv", True, 0
        for tl in self.items_tiles():
            for g, ti, nt, _ in tl:
                ok = (yield from self.wait_bar(self.pfull[g & 1], (g >> 1) & 1, who))
                if ok and ti == 0:
                    ok = yield from self.wait_bar(self.ofree, (oi & 1) ^ 1, who)
                for hh in range(2):
                    if not ok:
                        break
                    ok = yield from self.wait_bar(self.vfull[hh], g & 1, who)
                    if ok:
                        self.mma[who].append(self.vfree[hh])
                if not ok:
                    break
                self.mma[who].append(self.pdone[g & 1])
                if ti == nt - 1:
                    self.mma[who].append(self.odone)
            if not ok:
                break
            oi += 1
        self.mma[who].append(self.done)
        yield from self.drain_wait(self.done, 0)

    def kdeq(self):
        use = [0] * (TB * self.nrk)
        for tl in self.items_tiles():
            for g, ti, _, nb in tl:
                ok = yield from self.wait_bar(self.kfree[g & 1], ((g >> 1) & 1) ^ 1, "kdeq")
                if ok and ti == 0 and g > 0:
                    ok = yield from self.wait_bar(self.kfree[(g - 1) & 1], ((g - 1) >> 1) & 1, "kdeq")
                for jb in range(nb):
                    if not ok:
                        break
                    s = (g % self.nrk) * TB + jb
                    ok = yield from self.wait_bar(self.rkfull[s], use[s] & 1, "kdeq")
                if not ok:
                    return
                self.kfull[g & 1].arrive(128)
                for jb in range(nb):
                    s = (g % self.nrk) * TB + jb
                    self.rkfree[s].arrive(16)
                    use[s] += 1

    def vdeq(self, w):
        who, use = f"vdeq{w}", [[0] * self.nrv, [0] * self.nrv]
        for tl in self.items_tiles():
            for g, _, _, nb in tl:
                for hh in range(2):
                    jb = 4 * hh + w
                    ok = yield from self.wait_bar(self.vfree[hh], (g & 1) ^ 1, who)
                    if not ok:
                        return
                    if jb < nb:
                        st = g % self.nrv
                        ok = yield from self.wait_bar(self.rvfull[st * TB + jb], use[hh][st] & 1,
                                                      who)
                        if not ok:
                            return
                        use[hh][st] += 1
                        self.rvfree[st * TB + jb].arrive(32)
                    self.vfull[hh].arrive(32)

    def softmax(self, half):
        who, oi = f"soft{half}", 0
        for tl in self.items_tiles():
            for g, ti, nt, _ in tl:
                ok = (yield from self.wait_bar(self.sfull[g & 1], (g >> 1) & 1, who)) and \
                     (yield from self.wait_bar(self.pdone[g & 1], ((g >> 1) & 1) ^ 1, who))
                if ok and ti > 0 and ti % 3 == 1:
                    ok = yield from self.wait_bar(self.pdone[(g - 1) & 1], ((g - 1) >> 1) & 1, who)
                if not ok:
                    return
                self.sfree[g & 1].arrive(128)
                self.pfull[g & 1].arrive(128)
            ok = yield from self.wait_bar(self.odone, oi & 1, who)
            if not ok:
                return
            self.ofree.arrive(128)
            oi += 1

    # -- asynchronous engines
    def dma(self, rng):
        while True:
            if self.inflight:
                _, bar = self.inflight.pop(rng.randrange(len(self.inflight)))
                bar.arrive()
            yield lambda: True

    def mma_engine(self, who):
        while True:
            if self.mma[who]:
                self.mma[who].pop(0).arrive()
            yield lambda: True

    def run(self, seed):
        rng = random.Random(seed)
        roles = {f"prodK{j}": self.producer("K", j) for j in range(TB)}
        roles.update({f"prodV{j}": self.producer("V", j) for j in range(TB)})
        roles.update({"qk": self.qk(), "pv": self.pv(), "kdeq": self.kdeq(),
                      "soft0": self.softmax(0), "soft1": self.softmax(1)})
        roles.update({f"vdeq{w}": self.vdeq(w) for w in range(4)})
        engines = {"dma": self.dma(rng)}
        engines.update({f"mma_{w}": self.mma_engine(w) for w in self.mma})
        blocked = {a: None for a in roles}
        alive = set(roles)
        idle = 0
        while alive:
            progress = False
            order = sorted(alive)
            rng.shuffle(order)
            for a in order[: rng.randint(1, len(order))]:
                if blocked[a] is not None and not blocked[a]():
                    continue
                try:
                    blocked[a] = next(roles[a])
                except StopIteration:
                    alive.discard(a)
                progress = True
            if rng.random() < 0.5:
                for e in engines.values():
                    next(e)
            busy = self.inflight or any(self.mma.values())
            if not progress and not busy and all(blocked[a] is not None and not blocked[a]()
                                                for a in alive):
                idle += 1
                if idle > 3:
                    raise AssertionError(f"deadlock: {sorted(alive)}")
            else:
                idle = 0
        # every role has returned: the CTA exits and releases tensor memory
        assert not self.inflight, "copies in flight when the CTA exits"
        assert not any(self.mma.values()), "MMAs pending when tensor memory is released"
        return self.err


ITEMS = [[20, 3, 9, 1, 8, 64, 0, 5, 17], [40, 40, 40], [1, 1, 2, 3], [128, 7, 0, 64]]
ROLES = ["prodK0", "prodK5", "prodV3", "qk", "pv", "kdeq", "vdeq1", "vdeq3", "soft0", "soft1"]


@pytest.mark.parametrize("nrk,nrv", [(4, 2), (2, 1)])    # NVFP4 and FP8 ring sizes
@pytest.mark.parametrize("role", ROLES)
def test_one_expired_wait_ends_every_role_and_drains(nrk, nrv, role):
    fired = 0
    for items in ITEMS:
        for n in (0, 1, 3, 7):
            for seed in range(4):
                fired += AbortKernel(items, nrk, nrv, expire=(role, n)).run(seed)
    assert fired > 0, "the injected expiry never happened"


def test_no_expiry_runs_to_completion_without_the_flag():
    for items in ITEMS:
        for seed in range(6):
            assert not AbortKernel(items, 4, 2).run(seed)


def test_model_catches_a_fill_counted_before_its_stage_was_free():
    """The kernel once counted a fill before waiting for the stage; on an
    expired wait its drain then waited on the phase of a fill never issued,
    which reads as complete while the previous fill is still in flight."""
    with pytest.raises(AssertionError):
        for items in ITEMS:
            for n in range(6):
                for seed in range(12):
                    for role in ("prodK0", "prodK1", "prodV0"):
                        AbortKernel(items, 4, 2, expire=(role, n), count_before_wait=True).run(seed)
