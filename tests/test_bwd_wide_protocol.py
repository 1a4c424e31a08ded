"""Model of the wide-head backward's barrier protocol, run on random units and
random timings (CPU).

Above d = 128 the backward has three roles: a producer (unit fetch, K and V,
the ring of 64-column Q/dO chunks), an MMA issuer and the compute warps.  The
model runs each role as a coroutine that follows the kernel's loops and
parity expressions, lands TMA loads in any order, runs the tensor pipe's MMAs
and commits in issue order at random times, and checks every operand by
content: an MMA must read the chunk, the K/V tile, the P^T, dS^T or
accumulator it was issued for, and the compute warps must read the S^T, dP^T,
dQ or dV/dK they wait for.  TMEM regions are [0, 128) and [128, 256) (pass 1's
two S^T buffers; pass 2's S^T, dP^T, then dQ) and the dK/dV columns.

Pass 1 per unit: S(0), then S(s) and dV(s - 1), then dV(n - 1); the compute
warps turn S(s) into P(s).  Pass 2: S^T(s), dP^T(s), dS^T(s) by the compute
warps, dK(s), dQ(s), then the merge, which releases dQ's columns [0, 128)
before [128, 256).  Barriers follow mbarrier parity semantics (a wait whose
phase was overtaken is a hazard).  Planted mistakes must be caught.
"""
import random

import pytest


class Hazard(Exception):
    pass


class Bar:
    def __init__(self, count=1):
        self.count, self.pending, self.phases = count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.phases += 1

    def ready(self, parity, completion):
        """Hardware test of `parity`; `completion` (1-based) is the phase the
        caller means, to flag a wait whose phase was already overtaken."""
        if self.phases > completion:
            raise Hazard(f"phase {completion} overtaken ({self.phases} complete)")
        return (self.phases & 1) != parity


def run(units, C, slots, seed, mistake=None):
    """units: step counts per unit (query tiles, 0 allowed)."""
    rnd = random.Random(seed)
    B = lambda n=1: Bar(n)  # noqa: E731
    sched_full, sched_empty = [B(), B()], [B(2), B(2)]  # empty: MMA + compute
    kv_full, kv_empty = B(), B()
    slot_full, slot_free = [B() for _ in range(slots)], [B() for _ in range(slots)]
    s_full, p_ready, s_free = [B(), B()], [B(), B()], [B(), B()]
    sdp_full, ds_ready, dq_full, dq_free = B(), B(), B(), [B(), B()]
    dv_full, dk_full = B(), B()
    sched = [None, None]
    ring = [None] * slots
    mem = {"kv": None, "ds": None}
    tmem = {"lo": None, "hi": None, "acc": None}
    loads, pipe = [], []
    st = {"mma": 0}
    seq = list(enumerate(units))

    def wait(bar, parity, completion):
        while not bar.ready(parity, completion):
            yield

    # -------------------------------------------------------------- producer
    def producer():
        sched_it = unit_it = g = 0
        for u, ns in seq + [(-1, 0)]:
            slot = sched_it & 1
            n = sched_it >> 1
            yield from wait(sched_empty[slot], (n & 1) ^ 1, n)
            sched[slot] = (u, ns)
            sched_full[slot].arrive()
            sched_it += 1
            if u < 0:
                return
            if unit_it > 0:
                yield from wait(kv_empty, (unit_it - 1) & 1, unit_it)
            loads.append(("kv", u))
            unit_it += 1

            def chunk(what):
                nonlocal g
                sl, n = g % slots, g // slots
                if n > 0 and mistake != "no_slot_free_wait":
                    yield from wait(slot_free[sl], (n - 1) & 1, n)
                loads.append(("ring", sl, what))
                g += 1

            for s in range(ns + 1):
                if mistake == "producer_order" and s > 0:
                    for cc in range(C):
                        yield from chunk((u, 1, s - 1, "dO", cc))
                if s < ns:
                    for cc in range(C):
                        yield from chunk((u, 1, s, "Q", cc))
                if s > 0 and mistake != "producer_order":
                    for cc in range(C):
                        yield from chunk((u, 1, s - 1, "dO", cc))
            for s in range(ns):
                for kind in ("Q", "dO", "Q2"):
                    for cc in range(C):
                        yield from chunk((u, 2, s, kind, cc))

    # -------------------------------------------------------------- MMA issuer
    def mma():
        sched_it = unit_it = g = c1 = c2 = 0
        pend = {"lo": None, "hi": None}

        def settle(r):
            pd = pend[r]
            pend[r] = None
            if pd is not None:
                yield from wait(*pd)

        def expect(r, bar, parity, completion):
            yield from settle(r)
            pend[r] = (bar, parity, completion)

        def acquire(what):
            nonlocal g
            sl = g % slots
            yield from wait(slot_full[sl], (g // slots) & 1, g // slots + 1)
            return sl

        def release(sl):
            nonlocal g
            pipe.append(("commit", slot_free[sl]))
            g += 1

        def issue(reads, writes):
            pipe.append(("mma", reads, writes))

        # the first chunk's MMA overwrites (or starts accumulating into) the
        # region, the last one leaves the finished value
        def part(r, val, cc):
            return [(r, val if cc == C - 1 else ("partial",) + val)]

        while True:
            slot = sched_it & 1
            yield from wait(sched_full[slot], (sched_it >> 1) & 1, (sched_it >> 1) + 1)
            u, ns = sched[slot]
            sched_empty[slot].arrive()
            sched_it += 1
            if u < 0:
                break
            yield from wait(kv_full, unit_it & 1, unit_it + 1)
            unit_it += 1
            for s in range(ns + 1):
                if s < ns:
                    c = c1 + s
                    b = 0 if mistake == "single_s_buffer" else c & 1
                    r = ("lo", "hi")[b]
                    if mistake != "no_s_free":
                        yield from settle(r)
                    for cc in range(C):
                        sl = yield from acquire(None)
                        issue([("ring", sl, (u, 1, s, "Q", cc)), ("kv", None, ("kv", u))],
                              part(r, ("S", c), cc))
                        release(sl)
                    pipe.append(("commit", s_full[b]))
                if s > 0:
                    c = c1 + s - 1
                    b = 0 if mistake == "single_s_buffer" else c & 1
                    r = ("lo", "hi")[b]
                    par = ((c >> 1) & 1) ^ (1 if mistake == "wrong_p_ready_parity" else 0)
                    yield from wait(p_ready[b], par, (c >> 1) + 1)
                    for cc in range(C):
                        sl = yield from acquire(None)
                        prev = ("dV", u, s - 2) if s > 1 else None
                        issue([("ring", sl, (u, 1, s - 1, "dO", cc)), ("tmem", r, ("P", c))]
                              + ([("tmem", "acc", prev)] if prev and cc == 0 else []),
                              part("acc", ("dV", u, s - 1), cc))
                        release(sl)
                    pipe.append(("commit", s_free[b]))
                    if mistake == "no_s_free":
                        pend[r] = None
                    else:
                        yield from expect(r, s_free[b], (c >> 1) & 1, (c >> 1) + 1)
            c1 += ns
            if ns > 0 or mistake == "signal_empty_units":
                pipe.append(("commit", dv_full))
            for s in range(ns):
                c = c2 + s
                yield from settle("lo")
                for cc in range(C):
                    sl = yield from acquire(None)
                    issue([("ring", sl, (u, 2, s, "Q", cc)), ("kv", None, ("kv", u))],
                          part("lo", ("S2", c), cc))
                    release(sl)
                yield from settle("hi")
                for cc in range(C):
                    sl = yield from acquire(None)
                    issue([("ring", sl, (u, 2, s, "dO", cc)), ("kv", None, ("kv", u))],
                          part("hi", ("dP", c), cc))
                    release(sl)
                pipe.append(("commit", sdp_full))
                yield from wait(ds_ready, c & 1, c + 1)
                for cc in range(C):
                    sl = yield from acquire(None)
                    prev = ("dK", u, s - 1) if s > 0 else None
                    issue([("ring", sl, (u, 2, s, "Q2", cc)), ("ds", None, ("dS", c))]
                          + ([("tmem", "acc", prev)] if prev and cc == 0 else []),
                          part("acc", ("dK", u, s), cc))
                    release(sl)
                issue([("ds", None, ("dS", c)), ("kv", None, ("kv", u))],
                      [("lo", ("dQ", c)), ("hi", ("dQ", c))])
                pipe.append(("commit", dq_full))
                yield from expect("lo", dq_free[0], c & 1, c + 1)
                yield from expect("hi", dq_free[1], c & 1, c + 1)
            c2 += ns
            if ns > 0 or mistake == "signal_empty_units":
                pipe.append(("commit", dk_full))
            pipe.append(("commit", kv_empty))

    # -------------------------------------------------------------- compute
    def read(r, want):
        if tmem[r] != want:
            raise Hazard(f"compute read TMEM {r} = {tmem[r]}, expected {want}")

    def compute():
        sched_it = acc_it = c1 = c2 = 0
        late = None
        while True:
            slot = sched_it & 1
            yield from wait(sched_full[slot], (sched_it >> 1) & 1, (sched_it >> 1) + 1)
            u, ns = sched[slot]
            sched_empty[slot].arrive()
            sched_it += 1
            if u < 0:
                return
            for pss in range(2):
                for s in range(ns):
                    if pss == 0:
                        c = c1 + s
                        b = c & 1
                        yield from wait(s_full[b], (c >> 1) & 1, (c >> 1) + 1)
                        r = ("lo", "hi")[b]
                        read(r, ("S", c))
                        yield
                        tmem[r] = ("P", c)  # P^T over the S^T buffer
                        p_ready[b].arrive()
                        continue
                    c = c2 + s
                    yield from wait(sdp_full, c & 1, c + 1)
                    read("lo", ("S2", c))
                    read("hi", ("dP", c))
                    yield
                    mem["ds"] = ("dS", c)
                    ds_ready.arrive()
                    if late is not None and s == 0:
                        yield
                        read("acc", late)  # the dV epilogue, too late
                        late = None
                    yield from wait(dq_full, c & 1, c + 1)
                    if mistake == "dq_free_early":
                        dq_free[0].arrive()
                    yield  # the merge starts
                    read("lo", ("dQ", c))
                    yield  # columns [0, 128) of the merge
                    if mistake != "dq_free_early":
                        dq_free[0].arrive()
                    read("hi", ("dQ", c))
                    yield
                    dq_free[1].arrive()
                    mem["ds"] = ("stage", c)  # the merge's staging
                    yield
                if pss == 0:
                    c1 += ns
                else:
                    c2 += ns
                if ns > 0 or mistake == "signal_empty_units":
                    yield from wait(dv_full if pss == 0 else dk_full, acc_it & 1, acc_it + 1)
                if ns > 0:
                    want = ("dV", u, ns - 1) if pss == 0 else ("dK", u, ns - 1)
                    if mistake == "epilogue_late" and pss == 0:
                        late = want
                    else:
                        read("acc", want)
                yield
            if ns > 0 or mistake == "signal_empty_units":
                acc_it += 1

    # -------------------------------------------------------------- async units
    def execute(op):
        if op[0] == "commit":
            op[1].arrive()
            return
        _, reads, writes = op
        for kind, where, want in reads:
            have = ring[where] if kind == "ring" else (tmem[where] if kind == "tmem" else mem[kind])
            if have != want:
                raise Hazard(f"MMA read {kind} {where} = {have}, expected {want}")
        for r, val in writes:
            tmem[r] = val
        st["mma"] += 1

    def land(item):
        if item[0] == "kv":
            mem["kv"] = ("kv", item[1])
            kv_full.arrive()
        else:
            _, sl, what = item
            ring[sl] = what
            slot_full[sl].arrive()

    roles = [producer(), mma(), compute()]
    alive = [True] * 3
    for _ in range(2_000_000):
        if not any(alive) and not loads and not pipe:
            return st["mma"]
        r = rnd.random()
        if r < 0.25 and loads:
            land(loads.pop(rnd.randrange(len(loads))))
        elif r < 0.5 and pipe:
            execute(pipe.pop(0))
        else:
            k = rnd.randrange(3)
            if alive[k]:
                try:
                    next(roles[k])
                except StopIteration:
                    alive[k] = False
    raise Hazard("no progress (deadlock)")


def random_units(rnd):
    return [rnd.choice([0, 1, 2, 3, 5]) for _ in range(rnd.randint(1, 4))]


# (chunks per row, ring slots): d = 192 and d = 256
RINGS = [(3, 6), (4, 4)]


@pytest.mark.parametrize("C,slots", RINGS)
def test_protocol_is_hazard_and_deadlock_free(C, slots):
    for seed in range(150):
        units = random_units(random.Random(seed))
        n = run(units, C, slots, seed)
        # per step: pass 1 C + C MMA groups, pass 2 3C + one dQ
        assert n == sum(ns * (5 * C + 1) for ns in units)


# Each planted mistake must be caught:
# - no_slot_free_wait: a chunk loaded over one an MMA has yet to read;
# - producer_order: pass 1's dO(s - 1) loaded before Q(s), not in the MMAs' order;
# - no_s_free: S^T issued into a buffer whose P^T dV has yet to read;
# - single_s_buffer: pass 1 without the second S^T buffer;
# - wrong_p_ready_parity: dV issued on the wrong phase of p_ready;
# - dq_free_early: dQ's first columns released before the merge has read them;
# - epilogue_late: the dV epilogue moved after pass 2's first dS^T, so pass 2's
#   first dK may overwrite dV before it is read out;
# - signal_empty_units: dV/dK signalled for units without query tiles too, which
#   nothing of the compute warps paces, so the signals can overtake their waits.
MISTAKES = ["no_slot_free_wait", "producer_order", "no_s_free", "single_s_buffer",
            "wrong_p_ready_parity", "dq_free_early", "epilogue_late", "signal_empty_units"]


@pytest.mark.parametrize("C,slots", RINGS)
@pytest.mark.parametrize("mistake", MISTAKES)
def test_planted_mistakes_are_caught(mistake, C, slots):
    caught = False
    for seed in range(200):
        units = random_units(random.Random(seed))
        try:
            run(units, C, slots, seed, mistake=mistake)
        except Hazard:
            caught = True
            break
    assert caught, mistake
