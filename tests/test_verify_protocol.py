"""Model of the mbarrier hand-off protocol of the tcgen05 verify kernel
(csrc/pa_verify_umma.cuh), run under random schedules on the CPU.

Every role of the kernel is a generator that yields whenever it would wait on a
barrier; a barrier completes a phase after its count of arrivals, and a wait
for parity P passes once the phase with parity P has completed -- the
hardware's rule, under which a waiter that ran two phases ahead would pass on
a stale phase.  The roles log what they write and read, and the asserts check
the data flow itself: no buffer is read before it is written or overwritten
before its reader is done.  A wrong wait parity, a missing wait or a wrong
arrival count therefore fails an assert or deadlocks (both reported).

Roles (per CTA): K-side producer lanes 0-7 and V-side producer lanes 0-7
(block j of a tile), each side with its own ring of raw stages (stage =
(tile % rings) * 8 + j); the QK issuer; the PV issuer, which takes the V tile
in two half tiles of four blocks; the K dequant group; the four V dequant
warps (warp w dequantises block w of the first half tile, then block 4 + w of
the second); two softmax groups (half of the columns each).  Items are lists
of 16-token block counts; a tile is 8 blocks.
"""
import random

import pytest

TB = 8   # blocks per tile


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.completed = count, count, 0

    def arrive(self, n=1):
        self.pending -= n
        assert self.pending >= 0, "more arrivals than the barrier's count"
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def ready(self, parity):
        return (self.completed & 1) != parity


def tiles(n):
    return [min(TB, n - t * TB) for t in range((n + TB - 1) // TB)]


class Kernel:
    def __init__(self, items, nrk, nrv):
        self.items, self.nrk, self.nrv = items, nrk, nrv
        self.rkfull = [Bar(1) for _ in range(TB * nrk)]
        self.rkfree = [Bar(16) for _ in range(TB * nrk)]      # the block's 16 K rows
        self.rvfull = [Bar(1) for _ in range(TB * nrv)]
        self.rvfree = [Bar(32) for _ in range(TB * nrv)]      # 16 V rows, two threads each
        self.vfull = [Bar(128), Bar(128)]                     # every V thread, per half tile
        self.vfree = [Bar(1), Bar(1)]                         # the PV issuer, per half tile
        self.kfull = [Bar(128), Bar(128)]
        self.kfree = [Bar(1), Bar(1)]
        self.sfull = [Bar(1), Bar(1)]
        self.sfree = [Bar(256), Bar(256)]                     # both softmax groups
        self.pfull = [Bar(256), Bar(256)]
        self.pdone = [Bar(1), Bar(1)]                         # the PV issuer
        self.odone, self.ofree = Bar(1), Bar(256)
        self.log = set()

    @staticmethod
    def wait(bar, parity):
        while not bar.ready(parity):
            yield (bar, parity)

    def tiles_of_items(self, skip_empty=True):
        g = 0
        for n in self.items:
            if n == 0 and skip_empty:
                continue
            tl = tiles(n)
            for ti, nb in enumerate(tl):
                yield g, ti, len(tl), nb
                g += 1

    # -- producer lane j of one side
    def producer(self, side, j):
        nr = self.nrk if side == "K" else self.nrv
        full = self.rkfull if side == "K" else self.rvfull
        free = self.rkfree if side == "K" else self.rvfree
        use = [0] * nr
        last = {}   # stage -> tile of its previous fill
        for g, _, _, nb in self.tiles_of_items(skip_empty=False):
            if j >= nb:
                continue
            st = g % nr
            yield from self.wait(free[st * TB + j], (use[st] & 1) ^ 1)
            if st in last:   # the stage's previous tile was consumed
                assert ("read" + side, last[st], j) in self.log, "raw stage refilled before read"
            last[st] = g
            self.log.add(("fill" + side, g, j))
            full[st * TB + j].arrive()
            use[st] += 1

    def qk(self):
        for g, _, _, _ in self.tiles_of_items():
            yield from self.wait(self.kfull[g & 1], (g >> 1) & 1)
            yield from self.wait(self.sfree[g & 1], ((g >> 1) & 1) ^ 1)
            assert ("k", g) in self.log, "QK before its K tile was written"
            if g >= 2:
                assert ("s_read", g - 2, 0) in self.log and ("s_read", g - 2, 1) in self.log
            self.log.add(("qk", g))
            self.sfull[g & 1].arrive()
            self.kfree[g & 1].arrive()

    def pv(self):
        oi = 0
        for g, ti, nt, nb in self.tiles_of_items():
            yield from self.wait(self.pfull[g & 1], (g >> 1) & 1)
            if ti == 0:
                yield from self.wait(self.ofree, (oi & 1) ^ 1)
            assert ("p", g, 0) in self.log and ("p", g, 1) in self.log, "PV before P"
            for hh in range(2):
                yield from self.wait(self.vfull[hh], g & 1)
                for j in range(4 * hh, min(nb, 4 * hh + 4)):
                    assert ("v", g, j) in self.log, "PV before V"
                    assert ("v", g + 1, j) not in self.log, "V overwritten before PV read it"
                self.log.add(("pv", g, hh))
                self.vfree[hh].arrive()
            self.pdone[g & 1].arrive()
            if ti == nt - 1:
                self.odone.arrive()
                oi += 1

    def kdeq(self):
        use = [0] * (TB * self.nrk)
        for g, ti, _, nb in self.tiles_of_items():
            yield from self.wait(self.kfree[g & 1], ((g >> 1) & 1) ^ 1)
            if g >= 2:
                assert ("qk", g - 2) in self.log, "K tile overwritten before QK read it"
            if ti == 0 and g > 0:   # the q tile of a new item: the previous QK is done
                yield from self.wait(self.kfree[(g - 1) & 1], ((g - 1) >> 1) & 1)
                assert ("qk", g - 1) in self.log
            for jb in range(nb):
                s = (g % self.nrk) * TB + jb
                yield from self.wait(self.rkfull[s], use[s] & 1)
                assert ("fillK", g, jb) in self.log, "K dequant before its copy"
            self.log.add(("k", g))
            self.kfull[g & 1].arrive(128)
            for jb in range(nb):
                s = (g % self.nrk) * TB + jb
                self.log.add(("readK", g, jb))
                self.rkfree[s].arrive(16)
                use[s] += 1

    def vdeq(self, w):
        use = [[0] * self.nrv, [0] * self.nrv]
        for g, _, _, nb in self.tiles_of_items():
            for hh in range(2):
                jb = 4 * hh + w
                yield from self.wait(self.vfree[hh], (g & 1) ^ 1)
                if g >= 1:
                    assert ("pv", g - 1, hh) in self.log, "V half overwritten before PV read it"
                if jb < nb:
                    st = g % self.nrv
                    yield from self.wait(self.rvfull[st * TB + jb], use[hh][st] & 1)
                    assert ("fillV", g, jb) in self.log, "V dequant before its copy"
                    self.log.add(("v", g, jb))
                    self.log.add(("readV", g, jb))
                    self.rvfree[st * TB + jb].arrive(32)
                    use[hh][st] += 1
                self.vfull[hh].arrive(32)

    def softmax(self, half):
        oi = 0
        for g, ti, nt, _ in self.tiles_of_items():
            yield from self.wait(self.sfull[g & 1], (g >> 1) & 1)
            yield from self.wait(self.pdone[g & 1], ((g >> 1) & 1) ^ 1)
            assert ("qk", g) in self.log, "softmax before S"
            if g >= 2:   # the P buffer of tile g - 2 was read by both halves of PV
                assert ("pv", g - 2, 0) in self.log and ("pv", g - 2, 1) in self.log
            if ti > 0 and ti % 3 == 1:   # a redo: O^T is rescaled after PV(g - 1)
                yield from self.wait(self.pdone[(g - 1) & 1], ((g - 1) >> 1) & 1)
                assert ("pv", g - 1, 0) in self.log and ("pv", g - 1, 1) in self.log
            self.log.add(("s_read", g, half))
            self.log.add(("p", g, half))
            self.sfree[g & 1].arrive(128)
            self.pfull[g & 1].arrive(128)
            if ti == nt - 1:   # epilogue: O^T of the item after its last PV
                yield from self.wait(self.odone, oi & 1)
                self.ofree.arrive(128)
                oi += 1

    def run(self, seed):
        agents = {f"prodK{j}": self.producer("K", j) for j in range(TB)}
        agents.update({f"prodV{j}": self.producer("V", j) for j in range(TB)})
        agents.update({"qk": self.qk(), "pv": self.pv(), "kdeq": self.kdeq(),
                       "soft0": self.softmax(0), "soft1": self.softmax(1)})
        agents.update({f"vdeq{w}": self.vdeq(w) for w in range(4)})
        blocked = {a: None for a in agents}
        alive = set(agents)
        rng = random.Random(seed)
        while alive:
            progress = False
            order = sorted(alive)
            rng.shuffle(order)
            for a in order[: rng.randint(1, len(order))]:
                w = blocked[a]
                if w is not None and not w[0].ready(w[1]):
                    continue
                try:
                    blocked[a] = next(agents[a])
                except StopIteration:
                    alive.discard(a)
                progress = True
            if not progress and all(blocked[a] is not None and not blocked[a][0].ready(blocked[a][1])
                                    for a in alive):
                raise AssertionError(f"deadlock: {sorted(alive)}")


ITEM_MIXES = [
    [20, 3, 9, 1, 8, 64, 0, 5, 17],
    [9, 1, 8, 64, 0, 5, 17, 33],
    [1, 1, 1, 2, 3, 4, 5, 6, 7, 8, 9],
    [128, 7, 0, 0, 64],
    [40, 40, 40],
]


@pytest.mark.parametrize("nrk,nrv", [(4, 2), (2, 1), (3, 3)])   # NVFP4, FP8, and 3 + 3
@pytest.mark.parametrize("mix", range(len(ITEM_MIXES)))
def test_protocol_random_schedules(nrk, nrv, mix):
    for seed in range(12):
        Kernel(ITEM_MIXES[mix], nrk, nrv).run(seed)


def test_model_catches_a_missing_wait():
    """The model is not vacuous: a V dequant that skips its wait for the
    previous PV overwrites V before it is read."""
    class Broken(Kernel):
        def vdeq(self, w):
            use = [[0] * self.nrv, [0] * self.nrv]
            for g, _, _, nb in self.tiles_of_items():
                for hh in range(2):
                    jb = 4 * hh + w
                    if jb < nb:
                        st = g % self.nrv
                        yield from self.wait(self.rvfull[st * TB + jb], use[hh][st] & 1)
                        self.log.add(("v", g, jb))
                        self.rvfree[st * TB + jb].arrive(32)
                        use[hh][st] += 1
                    self.vfull[hh].arrive(32)

    with pytest.raises(AssertionError):
        for seed in range(40):
            Broken([40, 40, 40], 4, 2).run(seed)


def test_model_catches_a_missing_half_tile_wait():
    """A PV issuer that waits for the first half tile of V only reads the
    second half before its dequant wrote it (under some schedules)."""
    class Broken(Kernel):
        def pv(self):
            oi = 0
            for g, ti, nt, nb in self.tiles_of_items():
                yield from self.wait(self.pfull[g & 1], (g >> 1) & 1)
                if ti == 0:
                    yield from self.wait(self.ofree, (oi & 1) ^ 1)
                for hh in range(2):
                    if hh == 0:
                        yield from self.wait(self.vfull[hh], g & 1)
                    for j in range(4 * hh, min(nb, 4 * hh + 4)):
                        assert ("v", g, j) in self.log, "PV before V"
                    self.log.add(("pv", g, hh))
                    self.vfree[hh].arrive()
                self.pdone[g & 1].arrive()
                if ti == nt - 1:
                    self.odone.arrive()
                    oi += 1

    with pytest.raises(AssertionError):
        for seed in range(60):
            Broken([40, 40, 40], 4, 2).run(seed)
