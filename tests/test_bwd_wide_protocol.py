"""Model of the wide-head backward's load ring, run on random units and random
timings (CPU).

Above d = 128 one thread issues every TMA load and MMA of the backward, and
the 128 threads of the block meet at block barriers between the phases, so
the only pipelined hand-off is the ring of 64-column Q/dO chunks (4 slots at
d = 256, 6 at d = 192): the issuer loads a chunk into slot g % slots once the
MMA that read the slot's previous chunk has completed (slot_free, phase
g / slots - 1), and an MMA reads chunk g once its load has landed
(slot_full, phase g / slots), with loads issued up to slots - 1 chunks
ahead of the MMA that needs them, within the pass.  Pass 1 of a unit reads
per query tile Q then dO (C chunks each), pass 2 Q, dO, then Q again; the
ring's position carries over from pass to pass and unit to unit.

Barriers follow mbarrier parity semantics (a wait whose phase was overtaken
is a hazard), the tensor pipe runs MMAs and commits in issue order, TMA loads
land at random times.  Every MMA checks that its slot holds the chunk it
expects, and a load must never land in a slot whose previous chunk an issued
MMA has yet to read.  Planted mistakes must be caught.
"""
import random

import pytest



class Hazard(Exception):
    pass


class Bar:
    def __init__(self):
        self.phases = 0

    def ready(self, parity, completion):
        """Wait for the completion-th phase (1-based), by parity."""
        if self.phases > completion:
            raise Hazard(f"phase {completion} overtaken ({self.phases} complete)")
        return (self.phases & 1) != parity


def run(units, C, seed, slots, ahead, mistake=None):
    """units: list of step counts (query tiles per unit, 0 allowed)."""
    SLOTS = slots
    rnd = random.Random(seed)
    full = [Bar() for _ in range(SLOTS)]
    free = [Bar() for _ in range(SLOTS)]
    mma_done = Bar()
    slot = [None] * SLOTS          # chunk that landed in the slot
    pending_reads = [0] * SLOTS    # issued MMAs that still have to read the slot
    loads, pipe = [], []
    log = {"mma": 0}

    def chunk_of(u, pss, k, per):
        s, w = divmod(k, per)
        kind = "dO" if C <= w < 2 * C else "Q"
        return (u, pss, s, kind, w % C)

    def issuer():
        g0 = 0
        mma_waits = 0
        for u, ns in enumerate(units):
            for pss in range(2):
                per = 2 * C if pss == 0 else 3 * C
                total = ns * per
                issued = 0

                def issue_upto(kmax):
                    nonlocal issued
                    kmax = min(kmax, total)
                    while issued < kmax:
                        k = issued
                        g = g0 + k
                        sl, n = g % SLOTS, g // SLOTS
                        if n > 0 and mistake != "no_slot_free_wait":
                            par = ((n - 1) & 1) ^ (1 if mistake == "wrong_free_phase" else 0)
                            while not free[sl].ready(par, n):
                                yield
                        if pending_reads[sl]:
                            raise Hazard(f"load of chunk {g} into slot {sl} while an MMA still reads it")
                        loads.append((sl, chunk_of(u, pss, k, per)))
                        issued += 1

                def acquire(k):
                    yield from issue_upto(k + 1 + ahead)
                    g = g0 + k
                    while not full[g % SLOTS].ready((g // SLOTS) & 1, g // SLOTS + 1):
                        yield

                def mma(k):
                    sl = (g0 + k) % SLOTS
                    pending_reads[sl] += 1
                    pipe.append(("mma", sl, chunk_of(u, pss, k, per)))
                    pipe.append(("commit", free[sl]))

                for s in range(ns):
                    # S^T over the Q chunks (pass 2 also dP^T over the dO chunks)
                    for cc in range(C):
                        yield from acquire(s * per + cc)
                        mma(s * per + cc)
                    if pss == 1:
                        for cc in range(C):
                            yield from acquire(s * per + C + cc)
                            mma(s * per + C + cc)
                    pipe.append(("commit", mma_done))
                    while not mma_done.ready(mma_waits & 1, mma_waits + 1):
                        yield
                    mma_waits += 1
                    yield  # the block's P / dS phase
                    base = C if pss == 0 else 2 * C
                    for cc in range(C):  # dV (pass 1) or dK (pass 2)
                        yield from acquire(s * per + base + cc)
                        mma(s * per + base + cc)
                    pipe.append(("commit", mma_done))
                    while not mma_done.ready(mma_waits & 1, mma_waits + 1):
                        yield
                    mma_waits += 1
                g0 += total
        # drain
        while loads or pipe:
            yield

    def execute(op):
        if op[0] == "commit":
            op[1].phases += 1
            return
        _, sl, want = op
        if slot[sl] != want:
            raise Hazard(f"MMA read slot {sl} = {slot[sl]}, expected {want}")
        pending_reads[sl] -= 1
        log["mma"] += 1

    role = issuer()
    alive = True
    for _ in range(200000):
        if not alive and not loads and not pipe:
            return log["mma"]
        r = rnd.random()
        if r < 0.3 and loads:
            sl, chunk = loads.pop(rnd.randrange(len(loads)))  # loads land in any order
            slot[sl] = chunk
            full[sl].phases += 1
        elif r < 0.6 and pipe:
            execute(pipe.pop(0))
        elif alive:
            try:
                next(role)
            except StopIteration:
                alive = False
    raise Hazard("no progress (deadlock)")


def random_units(rnd):
    return [rnd.choice([0, 1, 2, 3, 5]) for _ in range(rnd.randint(1, 5))]


# (chunks per row, ring slots): d = 192 and d = 256
RINGS = [(3, 6), (4, 4)]


@pytest.mark.parametrize("C,slots", RINGS)
def test_ring_is_hazard_and_deadlock_free(C, slots):
    for seed in range(300):
        units = random_units(random.Random(seed))
        n = run(units, C, seed, slots, slots - 1)
        assert n == sum(ns * 5 * C for ns in units)  # 2C + 3C chunks per step, one MMA each


# Each planted mistake must be caught:
# - no_slot_free_wait: a load may land over a chunk an MMA has yet to read;
# - wrong_free_phase: waiting for the wrong completion of slot_free;
# - too_far_ahead: loads issued as many chunks ahead as there are slots.
@pytest.mark.parametrize("C,slots", RINGS)
@pytest.mark.parametrize("mistake", ["no_slot_free_wait", "wrong_free_phase", "too_far_ahead"])
def test_ring_planted_mistakes(mistake, C, slots):
    caught = False
    for seed in range(300):
        units = random_units(random.Random(seed))
        try:
            run(units, C, seed, slots, slots if mistake == "too_far_ahead" else slots - 1,
                mistake=None if mistake == "too_far_ahead" else mistake)
        except Hazard:
            caught = True
            break
    assert caught, mistake
