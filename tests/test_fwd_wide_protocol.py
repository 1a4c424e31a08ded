"""A model of the barrier protocol of the forward at head dimensions above 128,
run on random unit sequences and random timings.

The kernel's roles each become a generator that yields while it waits:

- the TMA producer (K one tile ahead of V, V in chunks over a ring of slots);
- the MMA issuer (S(j) into buffer j & 1, then PV(j-1) chunk by chunk);
- the softmax warps (S buffers alternating, P over S or in a region of its own);
- the epilogue warps (O stored from the row statistics the softmax warps hand over).

Barriers follow mbarrier semantics: a phase completes when its arrivals and
transaction bytes are in, and a wait on parity P returns while the current
phase's parity differs from P. The model flags every wait whose intended phase
has already been overtaken, since parity cannot tell those apart. The tensor
pipe runs MMAs and commits in issue order (a commit arrives once everything
issued before it has run). TMA loads complete at random times. Every MMA, load
and softmax step checks that the buffers it touches hold what it expects, and a
run that stops making progress is a deadlock.

Configurations: d = 256 (V in two 128-column chunks over 3 slots, P over its S
buffer) and d = 192 (whole V tiles over 2 slots, P in its own TMEM columns).
Planted mistakes in the protocol must be caught, so the checks have teeth.
"""
import random

import pytest


class Hazard(Exception):
    pass


class Barrier:
    def __init__(self, count):
        self.count, self.arrived, self.tx, self.phases = count, 0, 0, 0

    def arrive(self):
        self.arrived += 1
        self._complete()

    def expect_tx(self, tx):
        self.tx += tx
        self.arrive()

    def tx_done(self, tx):
        self.tx -= tx
        self._complete()

    def _complete(self):
        if self.arrived == self.count and self.tx == 0:
            self.phases += 1
            self.arrived = 0


def run(units, seed, nv, slots, sep_p, mistake=None):
    """units: list of (n, nkv): steps with MMAs, key/value tiles loaded."""
    rnd = random.Random(seed)
    bars = {}

    def bar(name, count=1):
        bars[name] = Barrier(count)

    for i in (0, 1):
        bar(f"sched_full{i}")
        bar(f"sched_empty{i}", 3)  # MMA issuer + softmax + epilogue warps
        bar(f"s_full{i}")
        bar(f"p_full{i}")
        bar(f"o_done{i}")
    for name in ("o_free", "q_full", "q_empty", "k_full", "k_empty", "ep_full"):
        bar(name)
    for i in range(slots):
        bar(f"v_full{i}")
        bar(f"v_empty{i}")

    def ready(name, parity, completion):
        """Wait for the completion-th phase (1-based) of a barrier, by parity."""
        b = bars[name]
        if b.phases > completion:
            raise Hazard(f"{name}: phase {completion} overtaken ({b.phases} complete)")
        return (b.phases & 1) != parity

    sched = [None, None]
    counter = [0]
    st = {"q": None, "k": None, "v": {}, "v_read": {}, "S": {}, "S_read": {}, "P": {},
          "O": [[] for _ in range(nv)], "stats": None, "out": []}
    loads, pipe = [], []

    def producer():
        it_sched = it_unit = k_it = v_it = 0
        while True:
            slot = it_sched & 1
            while not ready(f"sched_empty{slot}", ((it_sched >> 1) & 1) ^ 1, it_sched >> 1):
                yield
            u = counter[0]
            counter[0] += 1
            unit = (u,) + units[u] if u < len(units) else None
            sched[slot] = unit
            bars[f"sched_full{slot}"].arrive()
            it_sched += 1
            if unit is None:
                return
            uid, n, nkv = unit
            while not ready("q_empty", (it_unit & 1) ^ 1, it_unit):
                yield
            bars["q_full"].expect_tx(1 if n else 0)
            if n:
                loads.append(("q_full", "q", None, uid))
            it_unit += 1
            for j in range(nkv + 1):
                if j < nkv:
                    while not ready("k_empty", (k_it & 1) ^ 1, k_it):
                        yield
                    bars["k_full"].expect_tx(1)
                    loads.append(("k_full", "k", None, (uid, j)))
                    k_it += 1
                for h in range(nv if j >= 1 else 0):
                    s = v_it % slots
                    if mistake != "no_v_slot_wait":
                        while not ready(f"v_empty{s}", ((v_it // slots) & 1) ^ 1, v_it // slots):
                            yield
                    if s in st["v"] and not st["v_read"][s]:
                        raise Hazard(f"V slot {s} reloaded before its chunk was read")
                    st["v_read"][s] = False
                    bars[f"v_full{s}"].expect_tx(1)
                    loads.append((f"v_full{s}", "v", s, (uid, j - 1, h)))
                    v_it += 1
                yield

    def mma():
        it_sched = it_unit = g = k_it = v_it = ep = 0
        while True:
            slot = it_sched & 1
            while not ready(f"sched_full{slot}", (it_sched >> 1) & 1, (it_sched >> 1) + 1):
                yield
            unit = sched[slot]
            bars[f"sched_empty{slot}"].arrive()
            it_sched += 1
            if unit is None:
                return
            uid, n, nkv = unit
            while not ready("q_full", it_unit & 1, it_unit + 1):
                yield
            for j in range(nkv + 1):
                if j < nkv:
                    while not ready("k_full", k_it & 1, k_it + 1):
                        yield
                    if j < n:
                        gj = g + j
                        b = gj & 1
                        if not sep_p and gj >= 2 and mistake != "no_s_buffer_wait":
                            while not ready(f"o_done{b}", ((gj - 2) >> 1) & 1, ((gj - 2) >> 1) + 1):
                                yield
                        pipe.append(("S", (uid, j, b)))
                        pipe.append(("commit", f"s_full{b}"))
                    if j == nkv - 1:
                        pipe.append(("commit", "q_empty"))
                    pipe.append(("commit", "k_empty"))
                    k_it += 1
                if j >= 1:
                    jp = j - 1
                    gj = g + jp
                    b = gj & 1
                    if jp < n:
                        while not ready(f"p_full{b}", (gj >> 1) & 1, (gj >> 1) + 1):
                            yield
                        if jp == 0 and ep > 0:
                            while not ready("o_free", (ep - 1) & 1, ep):
                                yield
                    for h in range(nv):
                        s = v_it % slots
                        while not ready(f"v_full{s}", (v_it // slots) & 1, v_it // slots + 1):
                            yield
                        pipe.append(("PV", (uid, jp, b, h, s)) if jp < n else ("skip_v", s))
                        pipe.append(("commit", f"v_empty{s}"))
                        v_it += 1
                    if jp < n:
                        pipe.append(("commit", f"o_done{b}"))
                yield
            g += n
            it_unit += 1
            ep += n > 0

    def softmax():
        it_sched = it = ue = 0
        while True:
            slot = it_sched & 1
            while not ready(f"sched_full{slot}", (it_sched >> 1) & 1, (it_sched >> 1) + 1):
                yield
            unit = sched[slot]
            bars[f"sched_empty{slot}"].arrive()
            it_sched += 1
            if unit is None:
                return
            uid, n, _ = unit
            if n == 0:
                st["out"].append(("keyless", uid))
                continue
            for j in range(n):
                b = it & 1
                while not ready(f"s_full{b}", (it >> 1) & 1, (it >> 1) + 1):
                    yield
                if st["S"].get(b) != (uid, j):
                    raise Hazard(f"softmax ({uid},{j}) read S{b} = {st['S'].get(b)}")
                yield  # the exponentials
                if st["S"].get(b) != (uid, j):
                    raise Hazard("S overwritten while the softmax read it")
                st["S_read"][b] = True
                rescale = j > 0 and rnd.random() < 0.3
                if (sep_p or rescale) and it >= 1 and mistake != "no_pv_wait":
                    while not ready(f"o_done{(it - 1) & 1}", ((it - 1) >> 1) & 1, ((it - 1) >> 1) + 1):
                        yield
                p_at = "sep" if sep_p else b
                if st["P"].get(p_at) not in (None, "read"):
                    raise Hazard(f"P ({uid},{j}) written over unread P {st['P'][p_at]}")
                st["P"][p_at] = (uid, j)
                if rescale and any(o != [(uid, q) for q in range(j)] for o in st["O"]):
                    raise Hazard(f"rescale of ({uid},{j}) saw O = {st['O']}")
                bars[f"p_full{b}"].arrive()
                it += 1
                yield
            if ue > 0 and mistake != "no_stats_wait":
                while not ready("o_free", (ue - 1) & 1, ue):
                    yield
            st["stats"] = uid
            bars["ep_full"].arrive()
            ue += 1

    def epilogue():
        it_sched = it = ue = 0
        while True:
            slot = it_sched & 1
            while not ready(f"sched_full{slot}", (it_sched >> 1) & 1, (it_sched >> 1) + 1):
                yield
            unit = sched[slot]
            bars[f"sched_empty{slot}"].arrive()
            it_sched += 1
            if unit is None:
                return
            uid, n, _ = unit
            if n == 0:
                continue
            it += n
            while not ready("ep_full", ue & 1, ue + 1):
                yield
            while not ready(f"o_done{(it - 1) & 1}", ((it - 1) >> 1) & 1, ((it - 1) >> 1) + 1):
                yield
            ue += 1
            for _ in range(2):  # reads O and the statistics over a while
                if st["stats"] != uid:
                    raise Hazard(f"epilogue of {uid} read the statistics of {st['stats']}")
                if any(o != [(uid, q) for q in range(n)] for o in st["O"]):
                    raise Hazard(f"epilogue of {uid} read O = {st['O']}")
                yield
            st["out"].append(("stored", uid))
            bars["o_free"].arrive()

    def execute(op, arg):
        if op == "commit":
            bars[arg].arrive()
        elif op == "skip_v":
            st["v_read"][arg] = True
        elif op == "S":
            uid, j, b = arg
            if st["q"] != uid or st["k"] != (uid, j):
                raise Hazard(f"S ({uid},{j}) read Q {st['q']}, K {st['k']}")
            if st["S_read"].get(b) is False:
                raise Hazard(f"S ({uid},{j}) overwrote unread scores {st['S'][b]}")
            if not sep_p and st["P"].get(b) not in (None, "read"):
                raise Hazard(f"S ({uid},{j}) overwrote P {st['P'][b]} before PV read it")
            st["S"][b], st["S_read"][b] = (uid, j), False
            if not sep_p:
                st["P"][b] = None
        elif op == "PV":
            uid, j, b, h, s = arg
            p_at = "sep" if sep_p else b
            if st["v"].get(s) != (uid, j, h) or st["P"].get(p_at) != (uid, j):
                raise Hazard(f"PV ({uid},{j},{h}) read V {st['v'].get(s)}, P {st['P'].get(p_at)}")
            if j == 0:
                st["O"][h] = []
            st["O"][h].append((uid, j))
            st["v_read"][s] = True
            if h == nv - 1:
                st["P"][p_at] = "read"

    roles = [producer(), mma(), softmax(), epilogue()]
    alive = [True] * len(roles)
    for _ in range(400000):
        if not any(alive) and not pipe and not loads:
            break
        r = rnd.random()
        if r < 0.15 and loads:
            name, kind, slot, tag = loads.pop(rnd.randrange(len(loads)))
            if kind == "v":
                st["v"][slot] = tag
            else:
                st[kind] = tag
            bars[name].tx_done(1)
        elif r < 0.35 and pipe:
            execute(*pipe.pop(0))
        else:
            live = [i for i in range(len(roles)) if alive[i]]
            if live:
                i = rnd.choice(live)
                try:
                    next(roles[i])
                except StopIteration:
                    alive[i] = False
    else:
        raise Hazard("no progress (deadlock)")
    want = [("keyless", u) if units[u][0] == 0 else ("stored", u) for u in range(len(units))]
    if sorted(st["out"], key=lambda x: x[1]) != want:
        raise Hazard(f"outputs {st['out']}")


def random_units(rnd):
    """Causal-like step counts; n = 0 is a unit whose rows see no key (one
    key/value tile is still loaded and released)."""
    units = []
    for _ in range(rnd.randint(0, 7)):
        n = rnd.choice([0, 1, 1, 2, 3, 5, 8])
        units.append((n, max(n, 1)))
    return units


CONFIGS = {"d256": dict(nv=2, slots=3, sep_p=False), "d192": dict(nv=1, slots=2, sep_p=True)}


@pytest.mark.parametrize("cfg", sorted(CONFIGS))
def test_protocol_is_hazard_and_deadlock_free(cfg):
    for seed in range(400):
        rnd = random.Random(seed * 7 + 1)
        run(random_units(rnd), seed, **CONFIGS[cfg])


@pytest.mark.parametrize("cfg,mistake", [
    ("d256", "no_s_buffer_wait"),  # NOT caught: see below
    ("d256", "no_v_slot_wait"),
    ("d256", "no_pv_wait"),
    ("d256", "no_stats_wait"),
    ("d192", "no_v_slot_wait"),
    ("d192", "no_pv_wait"),
    ("d192", "no_stats_wait"),
])
def test_planted_mistakes_are_caught(cfg, mistake):
    caught = False
    for seed in range(400):
        rnd = random.Random(seed * 7 + 1)
        try:
            run(random_units(rnd), seed, mistake=mistake, **CONFIGS[cfg])
        except Hazard:
            caught = True
            break
    if mistake == "no_s_buffer_wait":
        # With an in-order tensor pipe, S(j) runs after PV(j-2) anyway; the
        # kernel keeps the wait because it does not rely on that order.
        assert not caught
    else:
        assert caught
