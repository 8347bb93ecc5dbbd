"""A host model of the forward megakernel's ring-buffer protocol, checked on the CPU.

The megakernel splits its co-resident CTAs in software ("Ring token buffers (macrobatch)"
and "Granularidade do overlap computacao-comunicacao" on the stamatios.com page). Gather
CTAs copy each macrobatch m into ring slot m mod S, row tile by row tile, and combine
finished macrobatches. GEMM CTAs run the up|gate tiles and then the down tiles of every
macrobatch, in one fixed task order. They signal through four kinds of counters:
gathered[m][r], hcnt[m][r], upg_done[m] and down_done[m].

The model replays that protocol as actors that each take their steps in order: the
gather CTAs, and the GEMM CTAs seen as one sequential step list each. The kernel's
producer warp may run ahead of its epilogue, which only allows more progress. A scheduler
interleaves the actors: at random, or always favouring one side. The tests check:

* every interleaving finishes (no deadlock);
* a slot is written only after every up|gate tile of the macrobatch that held it has read
  it, so no read sees another macrobatch's rows;
* a combine runs only after every down tile of its macrobatch;
* the test hook that withholds one row tile leaves every actor waiting (the kernel's
  bounded waits then end the launch with MOK_ERR_TIMEOUT), and no actor runs forever.

The step lists are derived from the kernel's loops and task order; the model shares no
code with the kernel.
"""
import random

import pytest


def row_tile(t, n_tiles):
    """Task t of a phase: row tile 2 (g // n_tiles) + (t & 1), with g = t // 2."""
    return ((t >> 1) // n_tiles) * 2 + (t & 1)


class RingModel:
    def __init__(self, mt, S, n_comm, G, n_up, n_down, withhold=False):
        self.mt, self.M, self.S = list(mt), len(mt), S
        self.n_comm, self.G, self.n_up, self.n_down = n_comm, G, n_up, n_down
        self.withhold = withhold
        self.gathered = {}
        self.hcnt = {}
        self.upg_done = [0] * self.M
        self.down_done = [0] * self.M
        self.slot = {}              # (slot, r) -> macrobatch whose rows it holds
        self.log = []
        self.actors = [self._comm(c) for c in range(n_comm)] + \
                      [self._gemm(g) for g in range(G)]

    # every actor is a generator of (condition, action) steps
    def _comm(self, c):
        M, S = self.M, self.S
        for m in range(M):
            if m >= S:
                need = self.mt[m - S] * self.n_up
                yield (lambda m=m, need=need: self.upg_done[m - S] >= need), None
            for r in range(c, self.mt[m], self.n_comm):
                yield (lambda: True), (lambda m=m, r=r: self._gather(m, r))
            if m >= 1:
                need = self.mt[m - 1] * self.n_down
                yield (lambda m=m, need=need: self.down_done[m - 1] >= need), \
                    (lambda m=m: self._combine(m - 1))
        yield from self._last_combine()

    def _gemm_tasks(self, g):
        base = 0
        for m in range(self.M):
            for ph in (0, 1):
                n_tiles = self.n_down if ph else self.n_up
                n = ((self.mt[m] + 1) // 2) * 2 * n_tiles
                t = (g - base) % self.G
                while t < n:
                    yield m, ph, t
                    t += self.G
                base = (base + n) % self.G

    def _gemm(self, g):
        for m, ph, t in self._gemm_tasks(g):
            n_tiles = self.n_down if ph else self.n_up
            r = row_tile(t, n_tiles)
            if r >= self.mt[m]:
                continue                                    # padding task: skipped
            if ph == 0:
                yield (lambda m=m, r=r: self.gathered.get((m, r), 0) >= 1), \
                    (lambda m=m, r=r: self._up_tile(m, r))
            else:
                yield (lambda m=m, r=r: self.hcnt.get((m, r), 0) >= self.n_up), \
                    (lambda m=m: self._down_tile(m))
        yield from self._last_combine()

    def _last_combine(self):
        m = self.M - 1
        need = self.mt[m] * self.n_down
        yield (lambda: self.down_done[m] >= need), (lambda: self._combine(m, last=True))

    # actions, with the safety checks
    def _gather(self, m, r):
        key = (m % self.S, r)
        prev = self.slot.get(key)
        if prev is not None:
            # the macrobatch that held the slot has had every up|gate tile read it
            assert self.upg_done[prev] == self.mt[prev] * self.n_up, (m, r, prev)
        self.slot[key] = m
        if not (self.withhold and m == 0 and r == 0):
            self.gathered[(m, r)] = self.gathered.get((m, r), 0) + 1

    def _up_tile(self, m, r):
        assert self.slot.get((m % self.S, r)) == m, (m, r)   # reads its own rows
        self.hcnt[(m, r)] = self.hcnt.get((m, r), 0) + 1
        self.upg_done[m] += 1

    def _down_tile(self, m):
        self.down_done[m] += 1

    def _combine(self, m, last=False):
        assert self.down_done[m] == self.mt[m] * self.n_down, m
        self.log.append(("combine", m))

    def run(self, pick):
        """Interleave the actors; ``pick(runnable)`` chooses the next one. Returns
        "done", or "blocked" when unfinished actors remain and none can move."""
        steps = [next(a, None) for a in self.actors]
        while True:
            live = [i for i, s in enumerate(steps) if s is not None]
            if not live:
                return "done"
            runnable = [i for i in live if steps[i][0]()]
            if not runnable:
                return "blocked"
            i = pick(runnable)
            act = steps[i][1]
            if act is not None:
                act()
            steps[i] = next(self.actors[i], None)


def _cases(n, seed):
    rnd = random.Random(seed)
    for _ in range(n):
        M = rnd.randint(1, 5)
        yield dict(mt=[rnd.randint(0, 5) for _ in range(M)], S=rnd.randint(1, M),
                   n_comm=rnd.randint(1, 3), G=rnd.randint(1, 4), n_up=rnd.randint(1, 3),
                   n_down=rnd.randint(1, 3))


PICKS = {
    "first": lambda rnd: (lambda r: r[0]),
    "last": lambda rnd: (lambda r: r[-1]),
    "random": lambda rnd: (lambda r: rnd.choice(r)),
}


@pytest.mark.parametrize("policy", sorted(PICKS))
def test_every_interleaving_finishes_and_reuses_slots_safely(policy):
    rnd = random.Random(7)
    for case in _cases(300, seed=11):
        for _ in range(3 if policy == "random" else 1):
            model = RingModel(**case)
            assert model.run(PICKS[policy](rnd)) == "done", case
            combines = [m for kind, m in model.log if kind == "combine"]
            # the gather CTAs combine 0 .. M-2 once each; every CTA combines M-1
            M = len(case["mt"])
            want = sorted([m for m in range(M - 1) for _ in range(case["n_comm"])] +
                          [M - 1] * (case["n_comm"] + case["G"]))
            assert sorted(combines) == want, case


def test_the_bench_and_test_shapes_finish():
    """The ring shapes the megakernel runs: the EP=64 slice's four macrobatches through
    three slots, and the ring test's four macrobatches through two slots, with the SM
    split the library picks and a few others."""
    rnd = random.Random(3)
    for mt, S in (([32, 32, 32, 32], 3), ([16, 16, 16, 15], 2), ([3, 0, 2, 1], 1)):
        for n_comm, G in ((1, 8), (3, 6), (8, 24)):
            for n_up, n_down in ((16, 56), (2, 2)):
                model = RingModel(mt, S, n_comm, G, n_up, n_down)
                assert model.run(lambda r: rnd.choice(r)) == "done"


def test_a_withheld_row_tile_blocks_instead_of_running_on():
    """With row tile 0 of macrobatch 0 never published, the up|gate tiles that need it
    cannot start and everything behind them waits: the model stops with every actor
    blocked, which on the GPU is where the bounded waits expire."""
    rnd = random.Random(5)
    for case in _cases(100, seed=13):
        if case["mt"][0] == 0:
            continue
        model = RingModel(**case, withhold=True)
        assert model.run(lambda r: rnd.choice(r)) == "blocked", case
        assert model.gathered.get((0, 0), 0) == 0


def test_the_slot_check_catches_an_early_reuse():
    """The model's safety check is live: a gather side that does not wait for the slot to
    drain (the upg_done wait removed) trips it on some interleaving."""
    class NoDrainWait(RingModel):
        def _comm(self, c):
            for cond, act in RingModel._comm(self, c):
                if act is None:
                    continue                                 # skip the drain wait
                yield cond, act

    tripped = False
    for case in _cases(200, seed=17):
        if len(case["mt"]) <= case["S"]:
            continue
        try:
            NoDrainWait(**case).run(lambda r: r[0])           # the gather side first
        except AssertionError:
            tripped = True
            break
    assert tripped
