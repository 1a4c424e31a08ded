"""A model of the backward kernel's barrier protocol (one CTA), run on random
unit sequences and random timings, with the harness of the forward's models.

The kernel's roles become generators:

- the K/V/Q producer: a key/value tile per unit, and a two-stage Q ring
  whose barrier also waits for the LSE and D rows the producer's lanes write;
- the dO producer (one stage);
- the MMA issuer, readiness-ordered as in the kernel: dP and dV in whichever
  order their inputs arrive, then dQ, the next S and dK;
- two compute warpgroups, one per half of the query columns: P^T over S^T in
  TMEM, then dS^T into shared memory;
- the dQ drain, which also stores dK and dV at the end of each unit.

Regions and the steps that may touch them:

- TMEM: S^T/P^T, dP^T, dQ (in dP's columns at d = 128), and the dK and dV
  accumulators.
- Shared memory: K, V, the Q stages with their rows, dO and dS^T.

Every MMA, load and compute step checks the contents it reads and that
nothing it overwrites is still unread. The model runs each warpgroup as one
actor, and also as four warps that arrive on their own, each owning a quarter
of the key rows. In that mode every barrier phase must hold arrivals for a
single step or unit. The deterministic mode's cross-CTA semaphores are
outside this model; the schedule tests cover their order.
"""
import random

import pytest

from test_fwd_protocol import Hazard, Sim


def run_bwd(units, seed, alias, mistake=None, warps=1):
    """units: list of ni, the query tiles each key/value unit walks (0: a key
    tile no query sees, as with unequal lengths).  warps: each compute
    warpgroup and the drain as one actor (1), or as four warps arriving on
    their own (4), each owning a quarter of the key rows."""
    parts = 2 * warps  # compute actors: query-column half x key-row quarter
    sim = Sim([(n,) for n in units], seed, consumers=3 + parts + warps - 1)
    for name in ("kv_full", "kv_empty", "do_full", "do_empty", "s_full", "dp_full", "s_free",
                 "dq_full", "dkv_full"):
        sim.bar(name)
    for name in ("p_ready", "ds_ready"):
        sim.bar(name, parts)
    for name in ("dq_free", "dkv_free"):
        sim.bar(name, warps)
    for s in (0, 1):
        sim.bar(f"q_full{s}", 2)  # the TMA bytes' arrival + the rows' arrival
        sim.bar(f"q_empty{s}")
    smem = {}
    everyone, drainers = set(range(parts)), set(range(warps))
    st = {"rows": {}, "rows_read": {}, "S": [None] * parts, "P_read": True, "dP": None,
          "dP_read": set(everyone), "dQ": None, "dQ_read": set(drainers), "dS": [None] * parts,
          "dS_read": 2, "dK": [], "dV": [], "dkv_read": set(drainers), "do_read": True,
          "kv_read": True, "q_read": {}}

    def producer():
        it_sched = it_unit = c = 0
        while True:
            unit = yield from sim.grab(it_sched)
            it_sched += 1
            if unit is None:
                return
            uid, ni = unit
            while not sim.ready("kv_empty", (it_unit & 1) ^ 1, it_unit):
                yield
            if not st["kv_read"]:
                raise Hazard(f"K/V of {uid} loaded over tiles still read")
            st["kv_read"] = False
            sim.bars["kv_full"].expect_tx(2)
            sim.issue("kv_full", "k", uid)
            sim.issue("kv_full", "v", uid)
            it_unit += 1
            for s in range(ni):
                q = c & 1
                if mistake != "no_q_empty_wait":
                    while not sim.ready(f"q_empty{q}", ((c >> 1) & 1) ^ 1, c >> 1):
                        yield
                if st["q_read"].get(q) is False or st["rows_read"].get(q, parts) != parts:
                    raise Hazard(f"Q stage {q} reloaded while still read")
                st["q_read"][q], st["rows_read"][q] = False, 0
                sim.load(f"q_full{q}", f"q{q}", (uid, s))
                st["rows"][q] = (uid, s)  # the lanes' LSE and D rows
                sim.bars[f"q_full{q}"].arrive()
                c += 1
                yield

    def do_producer():
        it_sched = c = 0
        while True:
            unit = yield from sim.take(it_sched)
            it_sched += 1
            if unit is None:
                return
            uid, ni = unit
            for s in range(ni):
                if mistake != "no_do_empty_wait":
                    while not sim.ready("do_empty", (c & 1) ^ 1, c):
                        yield
                if not st["do_read"]:
                    raise Hazard("dO reloaded before dP and dV read it")
                st["do_read"] = False
                sim.load("do_full", "do", (uid, s))
                c += 1
                yield

    def mma():
        it_sched = it_unit = cnt = 0
        held_dk = None  # the dk_after_next_dp mistake: dK(c) held back past dP(c+1)
        while True:
            unit = yield from sim.take(it_sched)
            it_sched += 1
            if unit is None:
                return
            uid, ni = unit
            while not sim.ready("kv_full", it_unit & 1, it_unit + 1):
                yield
            if ni > 0:
                while not sim.ready(f"q_full{cnt & 1}", (cnt >> 1) & 1, (cnt >> 1) + 1):
                    yield
                if cnt > 0 and mistake != "no_s_free_wait":
                    while not sim.ready("s_free", (cnt - 1) & 1, cnt):
                        yield
                sim.pipe += [("S", (uid, 0, cnt)), ("commit", "s_full")]
            for s in range(ni):
                q = cnt & 1
                while not sim.ready("do_full", cnt & 1, cnt + 1):
                    yield
                dp_done = dv_done = False
                while not (dp_done and dv_done):
                    if not dp_done and (not alias or cnt == 0 or mistake == "no_dq_free_wait"
                                        or sim.ready("dq_free", (cnt - 1) & 1, cnt)):
                        sim.pipe += [("dP", (uid, s)), ("commit", "dp_full")]
                        if held_dk:
                            sim.pipe += held_dk
                            held_dk = None
                        dp_done = True
                        continue
                    if not dv_done and sim.ready("p_ready", cnt & 1, cnt + 1) and (
                            s != 0 or it_unit == 0 or mistake == "no_dkv_free_wait"
                            or sim.ready("dkv_free", (it_unit - 1) & 1, it_unit)):
                        sim.pipe += [("dV", (uid, s)), ("commit", "s_free")]
                        dv_done = True
                        continue
                    yield
                sim.pipe += [("do_read", None), ("commit", "do_empty")]
                s_done, q_done, k_done = s + 1 >= ni, False, False
                while not (s_done and q_done and k_done):
                    if not q_done and sim.ready("ds_ready", cnt & 1, cnt + 1) and (
                            alias or cnt == 0 or sim.ready("dq_free", (cnt - 1) & 1, cnt)):
                        sim.pipe += [("dQ", (uid, s)), ("commit", "dq_full")]
                        q_done = True
                        continue
                    nq = (cnt + 1) & 1
                    if not s_done and sim.ready(f"q_full{nq}", ((cnt + 1) >> 1) & 1,
                                                ((cnt + 1) >> 1) + 1) and (
                            mistake == "no_s_free_wait" or sim.ready("s_free", cnt & 1, cnt + 1)):
                        sim.pipe += [("S", (uid, s + 1, cnt + 1)), ("commit", "s_full")]
                        s_done = True
                        continue
                    if not k_done and q_done:
                        ops = [("dK", (uid, s, q)), ("q_read", q), ("commit", f"q_empty{q}")]
                        if mistake == "dk_after_next_dp" and s + 1 < ni:
                            held_dk = ops
                        else:
                            sim.pipe += ops
                        k_done = True
                        continue
                    yield
                cnt += 1
            if ni == 0 and it_unit > 0 and mistake != "no_empty_unit_dkv_wait":
                # a unit no query sees issues no dV, whose first one waits for the
                # last epilogue: wait here, or dkv_full could run two phases ahead
                while not sim.ready("dkv_free", (it_unit - 1) & 1, it_unit):
                    yield
            sim.pipe += [("commit", "dkv_full"), ("kv_read", None), ("commit", "kv_empty")]
            it_unit += 1
            yield

    def compute(pt):
        it_sched = cnt = 0
        while True:
            unit = yield from sim.take(it_sched)
            it_sched += 1
            if unit is None:
                return
            uid, ni = unit
            for s in range(ni):
                q = cnt & 1
                while not sim.ready(f"q_full{q}", (cnt >> 1) & 1, (cnt >> 1) + 1):
                    yield
                while not sim.ready("s_full", cnt & 1, cnt + 1):
                    yield
                if st["S"][pt] != ("S", uid, s) or st["rows"].get(q) != (uid, s):
                    raise Hazard(f"compute {pt} ({uid},{s}) read {st['S'][pt]}, rows {st['rows'].get(q)}")
                yield  # P^T = exp2(S^T - LSE)
                st["S"][pt] = ("P", uid, s)
                sim.bars["p_ready"].arrive((uid, s))
                # dp_full(c) also covers dQ(c-1) and dK(c-1), the readers of the
                # last dS^T: the issuer puts both ahead of dP(c) on the in-order
                # pipe, so the kernel has no barrier of its own for them
                while not sim.ready("dp_full", cnt & 1, cnt + 1):
                    yield
                if st["dP"] != (uid, s) or st["rows"].get(q) != (uid, s):
                    raise Hazard(f"compute {pt} ({uid},{s}) read dP {st['dP']}")
                # this part's slice of the last complete dS^T tile must have been
                # read by both dQ and dK before it is overwritten
                if st["dS"][pt] is not None and st["dS_read"] != 2:
                    raise Hazard(f"dS of ({uid},{s}) written before dQ and dK read the last")
                yield  # dS^T = P^T (dP^T - D)
                if st["dP"] != (uid, s):
                    raise Hazard("dP overwritten while compute read it")
                st["dP_read"].add(pt)
                st["rows_read"][q] = st["rows_read"].get(q, 0) + 1
                st["dS"][pt] = (uid, s)
                if st["dS"] == [(uid, s)] * parts:
                    st["dS_read"] = 0
                sim.bars["ds_ready"].arrive((uid, s))
                cnt += 1

    def drain(w):
        it_sched = it_unit = cnt = 0
        while True:
            unit = yield from sim.take(it_sched)
            it_sched += 1
            if unit is None:
                return
            uid, ni = unit
            for s in range(ni):
                while not sim.ready("dq_full", cnt & 1, cnt + 1):
                    yield
                for _ in range(2):  # reads its dQ rows over a while
                    if st["dQ"] != (uid, s):
                        raise Hazard(f"drain warp {w} read dQ {st['dQ']}, expected {(uid, s)}")
                    yield
                st["dQ_read"].add(w)
                sim.bars["dq_free"].arrive((uid, s))
                cnt += 1
            while not sim.ready("dkv_full", it_unit & 1, it_unit + 1):
                yield
            want = [(uid, s) for s in range(ni)]
            for _ in range(2):
                if ni and (st["dK"] != want or st["dV"] != want):
                    raise Hazard(f"epilogue of {uid} read dK {st['dK']}, dV {st['dV']}")
                yield
            st["dkv_read"].add(w)
            if w == 0:
                sim.out.append(("stored", uid))
            sim.bars["dkv_free"].arrive(uid)
            it_unit += 1

    def execute(op, arg):
        if op == "commit":
            sim.bars[arg].arrive()
        elif op == "do_read":
            st["do_read"] = True
        elif op == "kv_read":
            st["kv_read"] = True
        elif op == "q_read":
            st["q_read"][arg] = True
        elif op == "S":
            uid, s, c = arg
            q = c & 1
            if smem.get(f"q{q}") != (uid, s) or smem.get("k") != uid:
                raise Hazard(f"S ({uid},{s}) read Q {smem.get(f'q{q}')}, K {smem.get('k')}")
            if not st["P_read"]:
                raise Hazard(f"S ({uid},{s}) overwrote P^T {st['S']} before dV read it")
            st["S"], st["P_read"] = [("S", uid, s)] * parts, False
        elif op == "dP":
            uid, s = arg
            if smem.get("v") != uid or smem.get("do") != (uid, s):
                raise Hazard(f"dP ({uid},{s}) read V {smem.get('v')}, dO {smem.get('do')}")
            if st["dP_read"] != everyone:
                raise Hazard(f"dP ({uid},{s}) overwrote dP {st['dP']} before compute read it")
            if alias and st["dQ_read"] != drainers:
                raise Hazard(f"dP ({uid},{s}) overwrote dQ {st['dQ']} before the drain read it")
            st["dP"], st["dP_read"] = (uid, s), set()
        elif op == "dV":
            uid, s = arg
            if st["S"] != [("P", uid, s)] * parts or smem.get("do") != (uid, s):
                raise Hazard(f"dV ({uid},{s}) read {st['S']}, dO {smem.get('do')}")
            if s == 0:
                if st["dkv_read"] != drainers:
                    raise Hazard(f"dV of {uid} reset before the epilogue read the last")
                st["dV"] = []
            st["dV"].append((uid, s))
            st["P_read"] = True
        elif op == "dQ":
            uid, s = arg
            if st["dS"] != [(uid, s)] * parts or smem.get("k") != uid:
                raise Hazard(f"dQ ({uid},{s}) read dS {st['dS']}")
            if st["dQ_read"] != drainers:
                raise Hazard(f"dQ ({uid},{s}) overwrote dQ {st['dQ']} before the drain read it")
            if alias and st["dP_read"] != everyone:
                raise Hazard(f"dQ ({uid},{s}) overwrote dP before compute read it")
            st["dQ"], st["dQ_read"] = (uid, s), set()
            if alias:
                st["dP"] = None  # its columns now hold dQ
            st["dS_read"] += 1
        elif op == "dK":
            uid, s, q = arg
            if st["dS"] != [(uid, s)] * parts or smem.get(f"q{q}") != (uid, s):
                raise Hazard(f"dK ({uid},{s}) read dS {st['dS']}, Q {smem.get(f'q{q}')}")
            if s == 0:
                st["dK"] = []
                st["dkv_read"] = set()  # both accumulators now hold this unit's
            st["dK"].append((uid, s))
            st["dS_read"] += 1

    roles = [producer(), do_producer(), mma()] + [compute(pt) for pt in range(parts)] + [
        drain(w) for w in range(warps)]
    sim.run(roles, execute, smem)
    if sorted(sim.out) != [("stored", u) for u in range(len(units))]:
        raise Hazard(f"outputs {sim.out}")


def random_units(rnd):
    """Key/value units of a causal walk (1..8 query tiles), and units no query
    sees (0), in random order."""
    return [rnd.choice([0, 1, 1, 2, 3, 5, 8]) for _ in range(rnd.randint(0, 6))]


@pytest.mark.parametrize("warps", [1, 4])
@pytest.mark.parametrize("alias", [True, False], ids=["d128", "d64"])
def test_bwd_protocol_is_hazard_and_deadlock_free(alias, warps):
    for seed in range(300 if warps == 1 else 150):
        run_bwd(random_units(random.Random(seed * 11 + 5)), seed, alias, warps=warps)


# Mistakes the model must catch (True), and waits it shows to be implied by
# others (False), which the kernel keeps all the same:
# - no_s_free_wait: with an in-order tensor pipe, S(c+1) runs after dV(c),
#   the last reader of P^T(c), which was issued before it.
# - dk_after_next_dp (caught): dK(c) held back until after dP(c+1).  The
#   compute warps write dS(c+1) once dp_full(c+1) completes, and take that as
#   proof that dK(c) has read dS(c); this issue order would break it.
# no_empty_unit_dkv_wait is the wait at the end of a unit no query sees: the
# model found it missing (two such units in a row put dkv_full two phases
# ahead of the epilogue warps).
BWD_MISTAKES = {"no_q_empty_wait": True, "no_do_empty_wait": True, "no_dq_free_wait": True,
                "no_dkv_free_wait": True, "dk_after_next_dp": True, "no_s_free_wait": False,
                "no_empty_unit_dkv_wait": True}


@pytest.mark.parametrize("warps", [1, 4])
@pytest.mark.parametrize("mistake", sorted(BWD_MISTAKES))
def test_bwd_planted_mistakes(mistake, warps):
    caught = False
    for seed in range(300):
        try:
            run_bwd(random_units(random.Random(seed * 11 + 5)), seed, True, mistake, warps)
        except Hazard:
            caught = True
            break
    assert caught == BWD_MISTAKES[mistake]
