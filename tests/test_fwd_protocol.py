"""Models of the forward kernel's barrier protocols, run on random unit
sequences and random timings.

Each role of the kernel becomes a generator that yields while it waits:

- the TMA producer;
- the MMA issuer;
- the softmax warps of each query tile;
- above d = 128, the epilogue warps.

Barriers follow mbarrier semantics. A phase completes when its arrivals and
transaction bytes are in. A wait on parity P returns while the current
phase's parity differs from P. The model flags every wait whose intended
phase has already been overtaken, since parity cannot tell those apart.

The tensor pipe runs MMAs and commits in issue order: a commit arrives once
everything issued before it has run. TMA loads complete at random times. Every
MMA, load and softmax step checks that the buffers it touches hold what it
expects. A run that stops making progress is a deadlock.

Layouts modelled:

- d <= 128: two query tiles per unit, a K/V ring of 2 or 4 stages, P written
  over S_t in two halves (keys [0, 64) and [64, 128)), each handed to the MMA
  issuer on its own so that PV_t runs in two halves, one O per tile.
- d = 256: one query tile, S double-buffered, K one tile ahead of V and
  released box by box (each 64-column box reloaded once the S MMAs over it
  are done), V in two 128-column chunks over 3 slots, P over its S buffer, O
  stored by the epilogue warps.
- d = 192: as d = 256 but with whole V tiles over 2 slots and P in TMEM
  columns of its own.

Both models also run their softmax (and epilogue) warpgroups as four warps
each, each arriving on its own and owning a quarter of the rows. Each
arrival carries the step or unit it stands for, and a phase that completes
with arrivals for two different ones is a hazard: a fast warp must never
arrive for its next step inside the phase its neighbours are completing.

Planted mistakes in each protocol must be caught, so the checks have teeth.
"""
import random

import pytest


class Hazard(Exception):
    pass


class Barrier:
    def __init__(self, count):
        self.count, self.arrived, self.tx, self.phases = count, 0, 0, 0
        self.tags = set()

    def arrive(self, tag=None):
        """tag: what the arrival stands for (a step, a unit); one phase must not
        mix arrivals for different ones."""
        self.arrived += 1
        if tag is not None:
            self.tags.add(tag)
            if len(self.tags) > 1:
                raise Hazard(f"one phase mixes arrivals for {sorted(self.tags)}")
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
            self.tags = set()


class Sim:
    """Barriers, TMA loads in flight, the in-order tensor pipe and the unit
    scheduler slots shared by the roles of one CTA."""

    def __init__(self, units, seed, consumers):
        self.units, self.rnd = units, random.Random(seed)
        self.bars, self.loads, self.pipe = {}, [], []
        self.sched, self.counter = [None, None], 0
        self.out = []
        for i in (0, 1):
            self.bar(f"sched_full{i}")
            self.bar(f"sched_empty{i}", consumers)

    def bar(self, name, count=1):
        self.bars[name] = Barrier(count)

    def ready(self, name, parity, completion):
        """Wait for the completion-th phase (1-based) of a barrier, by parity."""
        b = self.bars[name]
        if b.phases > completion:
            raise Hazard(f"{name}: phase {completion} overtaken ({b.phases} complete)")
        return (b.phases & 1) != parity

    def grab(self, it):
        """Producer side of the scheduler slots: the next unit, or None at the end."""
        slot = it & 1
        while not self.ready(f"sched_empty{slot}", ((it >> 1) & 1) ^ 1, it >> 1):
            yield
        u = self.counter
        self.counter += 1
        self.sched[slot] = (u,) + self.units[u] if u < len(self.units) else None
        self.bars[f"sched_full{slot}"].arrive()
        return self.sched[slot]

    def take(self, it):
        """Consumer side of the scheduler slots."""
        slot = it & 1
        while not self.ready(f"sched_full{slot}", (it >> 1) & 1, (it >> 1) + 1):
            yield
        unit = self.sched[slot]
        self.bars[f"sched_empty{slot}"].arrive()
        return unit

    def load(self, bar, key, tag):
        """Arrive with one tile's bytes expected, and issue its load."""
        self.bars[bar].expect_tx(1)
        self.issue(bar, key, tag)

    def issue(self, bar, key, tag):
        """A load whose bytes an earlier arrival already announced."""
        self.loads.append((bar, key, tag))

    def run(self, roles, execute, smem):
        alive = [True] * len(roles)
        for _ in range(400000):
            if not any(alive) and not self.pipe and not self.loads:
                return
            r = self.rnd.random()
            if r < 0.15 and self.loads:
                bar, key, tag = self.loads.pop(self.rnd.randrange(len(self.loads)))
                smem[key] = tag
                self.bars[bar].tx_done(1)
            elif r < 0.35 and self.pipe:
                execute(*self.pipe.pop(0))
            else:
                live = [i for i in range(len(roles)) if alive[i]]
                if live:
                    i = self.rnd.choice(live)
                    try:
                        next(roles[i])
                    except StopIteration:
                        alive[i] = False
        raise Hazard("no progress (deadlock)")


def check_outputs(sim, keyless):
    want = sorted(("keyless", u) if k else ("stored", u) for u, k in keyless)
    if sorted(sim.out) != want:
        raise Hazard(f"outputs {sorted(sim.out)}, expected {want}")


# ------------------------------------------------------------------ d <= 128

def run_two_tile(units, seed, stages, mistake=None, warps=1):
    """units: list of (n0, n1, nkv): key/value steps of query tiles 0 and 1 (0:
    past the end, or no row sees a key), and tiles loaded (>= 1).  warps: each
    tile's softmax warpgroup as one actor (1), or as four warps arriving on
    their own (4), each owning a quarter of the rows."""
    sim = Sim(units, seed, consumers=1 + 2 * warps)  # MMA issuer + the softmax warps
    for t in (0, 1):
        for name in ("s_full", "o_done"):
            sim.bar(f"{name}{t}")
        for name in ("p_full", "p_hi", "o_free"):
            sim.bar(f"{name}{t}", warps)
    for name in ("q_full", "q_empty"):
        sim.bar(name)
    for s in range(stages):
        for name in ("k_full", "v_full", "kv_empty"):
            sim.bar(f"{name}{s}")
    smem = {}
    st = {"S": {}, "P": {}, "O": {0: [], 1: []}, "kv_read": {}, "q_read": True}

    def producer():
        it_sched = it_unit = kv_it = 0
        while True:
            unit = yield from sim.grab(it_sched)
            it_sched += 1
            if unit is None:
                return
            uid, n0, n1, nkv = unit
            if mistake != "no_q_empty_wait":
                while not sim.ready("q_empty", (it_unit & 1) ^ 1, it_unit):
                    yield
            if not st["q_read"]:
                raise Hazard(f"Q of {uid} loaded over a Q still read")
            # one arrival for the unit, with the bytes of the tiles that see a key
            sim.bars["q_full"].expect_tx((n0 > 0) + (n1 > 0))
            for t, n in ((0, n0), (1, n1)):
                if n:
                    st["q_read"] = False
                    sim.issue("q_full", f"q{t}", uid)
            it_unit += 1
            for j in range(nkv):
                s = kv_it % stages
                if mistake != "no_kv_empty_wait":
                    while not sim.ready(f"kv_empty{s}", ((kv_it // stages) & 1) ^ 1, kv_it // stages):
                        yield
                if st["kv_read"].get(s) is False:
                    raise Hazard(f"stage {s} reloaded before it was read")
                st["kv_read"][s] = False
                sim.load(f"k_full{s}", f"k{s}", (uid, j))
                sim.load(f"v_full{s}", f"v{s}", (uid, j))
                kv_it += 1
                yield

    def mma():
        it_sched = it_unit = kv_it = 0
        it, ep = [0, 0], [0, 0]
        while True:
            unit = yield from sim.take(it_sched)
            it_sched += 1
            if unit is None:
                return
            uid, n0, n1, nkv = unit
            n = (n0, n1)
            while not sim.ready("q_full", it_unit & 1, it_unit + 1):
                yield
            for j in range(nkv):
                s, par = kv_it % stages, (kv_it // stages) & 1
                while not sim.ready(f"k_full{s}", par, kv_it // stages + 1):
                    yield
                for t in (0, 1):
                    if j >= n[t]:
                        continue
                    if it[t] > 0 and mistake != "no_s_wait":
                        while not sim.ready(f"o_done{t}", (it[t] - 1) & 1, it[t]):
                            yield
                    sim.pipe.append(("S", (uid, t, j, s)))
                    sim.pipe.append(("commit", f"s_full{t}"))
                if j == nkv - 1:
                    sim.pipe.append(("commit", "q_empty"))
                while not sim.ready(f"v_full{s}", par, kv_it // stages + 1):
                    yield
                for t in (0, 1):
                    if j >= n[t]:
                        continue
                    while not sim.ready(f"p_full{t}", it[t] & 1, it[t] + 1):
                        yield
                    if j == 0 and ep[t] > 0 and mistake != "no_o_free_wait":
                        while not sim.ready(f"o_free{t}", (ep[t] - 1) & 1, ep[t]):
                            yield
                    sim.pipe.append(("PV", (uid, t, j, s, 0)))  # keys [0, 64)
                    if mistake != "no_p_hi_wait":
                        while not sim.ready(f"p_hi{t}", it[t] & 1, it[t] + 1):
                            yield
                    sim.pipe.append(("PV", (uid, t, j, s, 1)))  # keys [64, 128)
                    sim.pipe.append(("commit", f"o_done{t}"))
                    it[t] += 1
                sim.pipe.append(("kv_read", s))
                sim.pipe.append(("commit", f"kv_empty{s}"))
                kv_it += 1
                yield
            it_unit += 1
            for t in (0, 1):
                ep[t] += n[t] > 0

    def softmax(t, w):
        it_sched = it = 0
        while True:
            unit = yield from sim.take(it_sched)
            it_sched += 1
            if unit is None:
                return
            uid, n0, n1, _ = unit
            nt = (n0, n1)[t]
            if nt == 0:
                continue
            for j in range(nt):
                while not sim.ready(f"s_full{t}", it & 1, it + 1):
                    yield
                if st["S"].get(t) != (uid, j):
                    raise Hazard(f"softmax {t}.{w} ({uid},{j}) read S = {st['S'].get(t)}")
                yield  # the row maximum (all of S_t is now in registers)
                if st["S"].get(t) != (uid, j):
                    raise Hazard("S overwritten while the softmax read it")
                done = [(uid, q, h) for q in range(j) for h in (0, 1)]
                rescale = j > 0 and sim.rnd.random() < 0.3
                if rescale and mistake != "rescale_after_p" and st["O"][t] != done:
                    raise Hazard(f"rescale of tile {t} ({uid},{j}) saw O = {st['O'][t]}")
                for hf, bar in ((0, "p_full"), (1, "p_hi")):
                    yield  # the exponentials of this half
                    st["P"].setdefault((t, hf), {})[w] = (uid, j)
                    sim.bars[f"{bar}{t}"].arrive((uid, j))
                    if hf == 0 and rescale and mistake == "rescale_after_p":
                        yield
                        if st["O"][t] != done:
                            raise Hazard(f"rescale of tile {t} ({uid},{j}) saw O = {st['O'][t]}")
                it += 1
                yield
            while not sim.ready(f"o_done{t}", (it - 1) & 1, it):
                yield
            for _ in range(2):  # reads O over a while
                if st["O"][t] != [(uid, q, h) for q in range(nt) for h in (0, 1)]:
                    raise Hazard(f"epilogue of tile {t} of {uid} read O = {st['O'][t]}")
                yield
            if w == 0:
                sim.out.append(("stored", (uid, t)))
            sim.bars[f"o_free{t}"].arrive(uid)

    def execute(op, arg):
        if op == "commit":
            if arg == "q_empty":
                st["q_read"] = True
            sim.bars[arg].arrive()
        elif op == "kv_read":
            st["kv_read"][arg] = True
        elif op == "S":
            uid, t, j, s = arg
            if smem.get(f"q{t}") != uid or smem.get(f"k{s}") != (uid, j):
                raise Hazard(f"S_{t} ({uid},{j}) read Q {smem.get(f'q{t}')}, K {smem.get(f'k{s}')}")
            for hf in (0, 1):
                if any(v != "read" for v in st["P"].get((t, hf), {}).values()):
                    raise Hazard(f"S_{t} ({uid},{j}) overwrote P {st['P'][(t, hf)]} before PV read it")
                st["P"][(t, hf)] = {}
            st["S"][t] = (uid, j)
        elif op == "PV":
            uid, t, j, s, hf = arg
            quarters = st["P"].get((t, hf), {})
            if smem.get(f"v{s}") != (uid, j) or len(quarters) != warps or any(
                    v != (uid, j) for v in quarters.values()):
                raise Hazard(f"PV_{t} ({uid},{j}) half {hf} read V {smem.get(f'v{s}')}, P {quarters}")
            if j == 0 and hf == 0:
                st["O"][t] = []
            st["O"][t].append((uid, j, hf))
            st["P"][(t, hf)] = {q: "read" for q in quarters}

    roles = [producer(), mma()] + [softmax(t, w) for t in (0, 1) for w in range(warps)]
    sim.run(roles, execute, smem)
    check_outputs(sim, [((u, t), units[u][t] == 0) for u in range(len(units)) for t in (0, 1)
                        if units[u][t] > 0])


def random_two_tile_units(rnd):
    """Causal units (tile 1 one step ahead of tile 0), non-causal ones, units
    past the end (no tile 1), and units of unequal query and key lengths whose
    first tile, or both, see no key (one K/V tile is still loaded)."""
    units = []
    for _ in range(rnd.randint(0, 6)):
        kind = rnd.choice(["causal", "dense", "tail", "keyless0", "keyless"])
        m = rnd.choice([0, 1, 2, 4])
        if kind == "causal":
            n0, n1 = 2 * m + 1, 2 * m + 2
        elif kind == "dense":
            n0 = n1 = m + 1
        elif kind == "tail":
            n0, n1 = 2 * m + 1, 0
        elif kind == "keyless0":
            n0, n1 = 0, m + 1
        else:
            n0 = n1 = 0
        units.append((n0, n1, max(n0, n1, 1)))
    return units


@pytest.mark.parametrize("warps", [1, 4])
@pytest.mark.parametrize("stages", [2, 4])
def test_two_tile_protocol_is_hazard_and_deadlock_free(stages, warps):
    for seed in range(300 if warps == 1 else 150):
        run_two_tile(random_two_tile_units(random.Random(seed * 7 + 3)), seed, stages,
                     warps=warps)


# Mistakes the model must catch (True), and waits it shows to be implied by
# others (False), which the kernel keeps all the same:
# - no_s_wait: with an in-order tensor pipe S_t(j) runs after PV_t(j-1)
#   anyway; the kernel does not rely on that order.
# - no_o_free_wait: the warpgroup that stores O_t is the one whose next P_t
#   the first PV_t of the next unit waits for.
# - no_p_hi_wait: PV_t's second half issued without waiting for the second
#   half of P;
# - rescale_after_p: the O~ rescale done after the first half of P is handed
#   over, when PV_t's first half may already be adding into O.
TWO_TILE_MISTAKES = {"no_s_wait": False, "no_o_free_wait": False, "no_kv_empty_wait": True,
                     "no_q_empty_wait": True, "no_p_hi_wait": True, "rescale_after_p": True}


@pytest.mark.parametrize("warps", [1, 4])
@pytest.mark.parametrize("mistake", sorted(TWO_TILE_MISTAKES))
def test_two_tile_planted_mistakes(mistake, warps):
    caught = False
    for seed in range(300):
        try:
            run_two_tile(random_two_tile_units(random.Random(seed * 7 + 3)), seed, 2, mistake,
                         warps)
        except Hazard:
            caught = True
            break
    assert caught == TWO_TILE_MISTAKES[mistake]


# ------------------------------------------------------------------ d > 128

def run_one_tile(units, seed, nv, slots, sep_p, nb, mistake=None, warps=1):
    """units: list of (n, nkv): steps with MMAs (0: no row sees a key), and
    key/value tiles loaded (>= 1).  nb: 64-column boxes of a K tile.  warps:
    the softmax and the epilogue warpgroups as one actor each (1), or as four
    warps arriving on their own (4), each owning a quarter of the rows."""
    sim = Sim(units, seed, consumers=1 + 2 * warps)  # MMA issuer + softmax + epilogue warps
    for i in (0, 1):
        sim.bar(f"s_full{i}")
        sim.bar(f"o_done{i}")
        sim.bar(f"p_full{i}", warps)  # P's first half (keys [0, 64))
        sim.bar(f"p_hi{i}", warps)    # P's second half
    for name in ["q_full", "q_empty", "k_full"] + [f"k_empty{c}" for c in range(nb)]:
        sim.bar(name)
    for name in ("o_free", "ep_full"):
        sim.bar(name, warps)
    for i in range(slots):
        sim.bar(f"v_full{i}")
        sim.bar(f"v_empty{i}")
    smem = {}
    st = {"v_read": {}, "S": {}, "S_read": {}, "P": {}, "O": [[] for _ in range(nv)],
          "stats": {}}

    def producer():
        it_sched = it_unit = k_it = v_it = 0
        while True:
            unit = yield from sim.grab(it_sched)
            it_sched += 1
            if unit is None:
                return
            uid, n, nkv = unit
            while not sim.ready("q_empty", (it_unit & 1) ^ 1, it_unit):
                yield
            if n:
                sim.load("q_full", "q", uid)
            else:
                sim.bars["q_full"].arrive()
            it_unit += 1
            for j in range(nkv + 1):
                if j < nkv:
                    if mistake == "k_arm_early":
                        sim.bars["k_full"].expect_tx(nb)
                    for c in range(nb):
                        if c == 0 or mistake != "no_k_box_wait":
                            while not sim.ready(f"k_empty{c}", (k_it & 1) ^ 1, k_it):
                                yield
                        if c == 0 and mistake != "k_arm_early":
                            # armed once the previous tile's phase is complete
                            sim.bars["k_full"].expect_tx(nb)
                        sim.issue("k_full", f"k{c}", (uid, j))
                        yield
                    k_it += 1
                for h in range(nv if j >= 1 else 0):
                    s = v_it % slots
                    if mistake != "no_v_slot_wait":
                        while not sim.ready(f"v_empty{s}", ((v_it // slots) & 1) ^ 1, v_it // slots):
                            yield
                    if st["v_read"].get(s) is False:
                        raise Hazard(f"V slot {s} reloaded before its chunk was read")
                    st["v_read"][s] = False
                    sim.load(f"v_full{s}", f"v{s}", (uid, j - 1, h))
                    v_it += 1
                yield

    def mma():
        it_sched = it_unit = g = k_it = v_it = ep = 0
        while True:
            unit = yield from sim.take(it_sched)
            it_sched += 1
            if unit is None:
                return
            uid, n, nkv = unit
            while not sim.ready("q_full", it_unit & 1, it_unit + 1):
                yield
            for j in range(nkv + 1):
                if j < nkv:
                    while not sim.ready("k_full", k_it & 1, k_it + 1):
                        yield
                    if j < n:
                        gj = g + j
                        b = gj & 1
                        if not sep_p and gj >= 2 and mistake != "no_s_buffer_wait":
                            while not sim.ready(f"o_done{b}", ((gj - 2) >> 1) & 1, ((gj - 2) >> 1) + 1):
                                yield
                        for c in range(nb):
                            if mistake == "k_box_release_early":
                                sim.pipe.append(("commit", f"k_empty{c}"))
                            sim.pipe.append(("S", (uid, j, b, c)))
                            if mistake != "k_box_release_early":
                                sim.pipe.append(("commit", f"k_empty{c}"))
                        sim.pipe.append(("commit", f"s_full{b}"))
                    else:
                        for c in range(nb):
                            sim.pipe.append(("commit", f"k_empty{c}"))
                    if j == nkv - 1:
                        sim.pipe.append(("commit", "q_empty"))
                    k_it += 1
                if j >= 1:
                    jp = j - 1
                    gj = g + jp
                    b = gj & 1
                    if jp < n:
                        while not sim.ready(f"p_full{b}", (gj >> 1) & 1, (gj >> 1) + 1):
                            yield
                        if jp == 0 and ep > 0 and mistake != "no_o_free_wait":
                            while not sim.ready("o_free", (ep - 1) & 1, ep):
                                yield
                    for h in range(nv):
                        s = v_it % slots
                        while not sim.ready(f"v_full{s}", (v_it // slots) & 1, v_it // slots + 1):
                            yield
                        if jp < n:
                            # the first chunk waits for P's second half halfway
                            sim.pipe.append(("PV", (uid, jp, b, h, s, 0)))
                            if h == 0 and mistake != "no_p_hi_wait":
                                while not sim.ready(f"p_hi{b}", (gj >> 1) & 1, (gj >> 1) + 1):
                                    yield
                            sim.pipe.append(("PV", (uid, jp, b, h, s, 1)))
                        else:
                            sim.pipe.append(("skip_v", s))
                        sim.pipe.append(("commit", f"v_empty{s}"))
                        v_it += 1
                    if jp < n:
                        sim.pipe.append(("commit", f"o_done{b}"))
                yield
            g += n
            it_unit += 1
            ep += n > 0

    def softmax(w):
        it_sched = it = ue = 0
        while True:
            unit = yield from sim.take(it_sched)
            it_sched += 1
            if unit is None:
                return
            uid, n, _ = unit
            if n == 0:
                if w == 0:
                    sim.out.append(("keyless", uid))
                continue
            for j in range(n):
                b = it & 1
                while not sim.ready(f"s_full{b}", (it >> 1) & 1, (it >> 1) + 1):
                    yield
                if st["S"].get(b) != (uid, j):
                    raise Hazard(f"softmax warp {w} ({uid},{j}) read S{b} = {st['S'].get(b)}")
                yield  # the row maximum (all of S is now in registers)
                if st["S"].get(b) != (uid, j):
                    raise Hazard("S overwritten while the softmax read it")
                st["S_read"].setdefault(b, set()).add(w)
                rescale = j > 0 and sim.rnd.random() < 0.3
                pv_done = it == 0
                done = [(uid, q, hf) for q in range(j) for hf in (0, 1)]
                if rescale:
                    # O~ first: PV(j - 1) done (S(j) may have finished before it)
                    if mistake != "no_pv_wait":
                        while not sim.ready(f"o_done{(it - 1) & 1}", ((it - 1) >> 1) & 1, ((it - 1) >> 1) + 1):
                            yield
                    pv_done = True
                    if any(o != done for o in st["O"]):
                        raise Hazard(f"rescale of ({uid},{j}) saw O = {st['O']}")
                p_at = "sep" if sep_p else b
                for hf, bar in ((0, "p_full"), (1, "p_hi")):
                    yield  # the exponentials of this half
                    if sep_p and not pv_done and mistake != "no_pv_wait":
                        # P has a region of its own: PV(j - 1) must have read it
                        while not sim.ready(f"o_done{(it - 1) & 1}", ((it - 1) >> 1) & 1, ((it - 1) >> 1) + 1):
                            yield
                        pv_done = True
                    mine = st["P"].setdefault((p_at, hf), {})
                    if mine.get(w) not in (None, "read"):
                        raise Hazard(f"P ({uid},{j}) half {hf} of warp {w} written over unread P {mine[w]}")
                    mine[w] = (uid, j)
                    sim.bars[f"{bar}{b}"].arrive((uid, j))
                it += 1
                yield
            if ue > 0 and mistake != "no_stats_wait":
                while not sim.ready("o_free", (ue - 1) & 1, ue):
                    yield
            st["stats"][w] = uid
            sim.bars["ep_full"].arrive(uid)
            ue += 1

    def epilogue(w):
        it_sched = it = ue = 0
        while True:
            unit = yield from sim.take(it_sched)
            it_sched += 1
            if unit is None:
                return
            uid, n, _ = unit
            if n == 0:
                continue
            it += n
            while not sim.ready("ep_full", ue & 1, ue + 1):
                yield
            while not sim.ready(f"o_done{(it - 1) & 1}", ((it - 1) >> 1) & 1, ((it - 1) >> 1) + 1):
                yield
            ue += 1
            for _ in range(2):  # reads O and the statistics of its rows over a while
                if st["stats"].get(w) != uid:
                    raise Hazard(f"epilogue warp {w} of {uid} read the statistics of {st['stats'].get(w)}")
                if any(o != [(uid, q, hf) for q in range(n) for hf in (0, 1)] for o in st["O"]):
                    raise Hazard(f"epilogue of {uid} read O = {st['O']}")
                yield
            if w == 0:
                sim.out.append(("stored", uid))
            sim.bars["o_free"].arrive(uid)

    def execute(op, arg):
        if op == "commit":
            sim.bars[arg].arrive()
        elif op == "skip_v":
            st["v_read"][arg] = True
        elif op == "S":
            # the MMAs over K's box c (the first one starts overwriting S_b)
            uid, j, b, c = arg
            if smem.get("q") != uid or smem.get(f"k{c}") != (uid, j):
                raise Hazard(f"S ({uid},{j}) box {c} read Q {smem.get('q')}, K {smem.get(f'k{c}')}")
            if c == 0:
                if b in st["S"] and len(st["S_read"].get(b, ())) < warps:
                    raise Hazard(f"S ({uid},{j}) overwrote unread scores {st['S'][b]}")
                for hf in (0, 1):
                    if not sep_p and any(v != "read" for v in st["P"].get((b, hf), {}).values()):
                        raise Hazard(f"S ({uid},{j}) overwrote P {st['P'][(b, hf)]} before PV read it")
                    if not sep_p:
                        st["P"][(b, hf)] = {}
            st["S"][b] = (uid, j) if c == nb - 1 else ("partial", uid, j)
            st["S_read"][b] = set()
        elif op == "PV":
            uid, j, b, h, s, hf = arg
            p_at = "sep" if sep_p else b
            quarters = st["P"].get((p_at, hf), {})
            if smem.get(f"v{s}") != (uid, j, h) or len(quarters) != warps or any(
                    v != (uid, j) for v in quarters.values()):
                raise Hazard(f"PV ({uid},{j},{h}) half {hf} read V {smem.get(f'v{s}')}, P {quarters}")
            if j == 0 and hf == 0:
                st["O"][h] = []
            st["O"][h].append((uid, j, hf))
            if hf == 1:
                st["v_read"][s] = True
            if h == nv - 1:
                st["P"][(p_at, hf)] = {w: "read" for w in quarters}

    roles = [producer(), mma()] + [softmax(w) for w in range(warps)] + [
        epilogue(w) for w in range(warps)]
    sim.run(roles, execute, smem)
    check_outputs(sim, [(u, units[u][0] == 0) for u in range(len(units))])


def random_one_tile_units(rnd):
    """Causal-like step counts; n = 0 is a unit whose rows see no key (one
    key/value tile is still loaded and released)."""
    units = []
    for _ in range(rnd.randint(0, 7)):
        n = rnd.choice([0, 1, 1, 2, 3, 5, 8])
        units.append((n, max(n, 1)))
    return units


ONE_TILE = {"d256": dict(nv=2, slots=3, sep_p=False, nb=4),
            "d192": dict(nv=1, slots=2, sep_p=True, nb=3)}


@pytest.mark.parametrize("warps", [1, 4])
@pytest.mark.parametrize("cfg", sorted(ONE_TILE))
def test_one_tile_protocol_is_hazard_and_deadlock_free(cfg, warps):
    for seed in range(400 if warps == 1 else 200):
        run_one_tile(random_one_tile_units(random.Random(seed * 7 + 1)), seed, warps=warps,
                     **ONE_TILE[cfg])


# As above; no_s_buffer_wait is implied by an in-order tensor pipe (S(j)
# runs after PV(j-2) anyway), which the kernel does not rely on.  Here the
# epilogue warps store O, so the first PV of a unit must wait for them.
# no_k_box_wait: K's boxes after the first loaded without waiting for their
# release; k_box_release_early: a box released before its S MMAs; k_arm_early:
# k_full armed for the next tile before the first box is free, possibly
# inside the phase of the tile still landing.
ONE_TILE_MISTAKES = {"no_s_buffer_wait": False, "no_v_slot_wait": True, "no_pv_wait": True,
                     "no_stats_wait": True, "no_o_free_wait": True, "no_k_box_wait": True,
                     "k_box_release_early": True, "k_arm_early": True, "no_p_hi_wait": True}


@pytest.mark.parametrize("warps", [1, 4])
@pytest.mark.parametrize("cfg", sorted(ONE_TILE))
@pytest.mark.parametrize("mistake", sorted(ONE_TILE_MISTAKES))
def test_one_tile_planted_mistakes(cfg, mistake, warps):
    if cfg == "d192" and mistake == "no_s_buffer_wait":
        pytest.skip("d = 192 has no such wait (P has columns of its own)")
    caught = False
    for seed in range(400):
        try:
            run_one_tile(random_one_tile_units(random.Random(seed * 7 + 1)), seed,
                         mistake=mistake, warps=warps, **ONE_TILE[cfg])
        except Hazard:
            caught = True
            break
    assert caught == ONE_TILE_MISTAKES[mistake]
