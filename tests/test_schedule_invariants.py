"""Deterministic-mode dQ ordering: invariants of the schedule, checked on the
CPU for many geometries (dense and packed, equal and different query/key
lengths, causal and not).

The backward's deterministic mode adds each dQ tile's contributions in a
fixed order enforced by one semaphore per tile: unit (key/value tile j)
waits until the semaphore equals its rank, then adds and increments it.
That is deadlock-free at any size only if, for every dQ tile,
  1. the ranks of its contributors are exactly 0, 1, ..., n-1, and
  2. every contributor with a lower rank was taken from the work counter
     earlier (so it is running or done, whatever CTA holds which unit).
This test restates the schedule (the scheduler's descending key/value-tile
order, each unit's walk and rank) from its definition in the kernels'
comments and checks both properties.  An earlier cyclic non-causal order
broke property 2.  A unit may walk a run of C query heads of one key/value
head, one after the other; the properties must hold for every run length.
"""
import itertools
import random

import pytest

TILE = 128


def cdiv(a, b):
    return -(-a // b)


def floor_div(a, b):
    return a // b  # Python floors


def unit_order(lk_list, H):
    """Deterministic order: key/value tile index descending across sequences
    (level order of the scheduler), sequences ranked by tile count descending
    (ties by index), heads innermost."""
    nt = [cdiv(L, TILE) for L in lk_list]
    ranked = sorted(range(len(lk_list)), key=lambda b: (-nt[b], b))
    maxnt = max(nt) if nt else 0
    order = []
    for m in range(maxnt - 1, -1, -1):
        for b in ranked:
            if nt[b] > m:
                for h in range(H):
                    order.append((b, m, h))
    return order


def unit_geometry(j, lq, lk, causal):
    nt = cdiv(lq, TILE)
    ntk = cdiv(lk, TILE)
    off = lk - lq
    i0 = max(0, floor_div(j * TILE - off, TILE)) if causal else 0
    ni = max(0, nt - i0)
    return nt, ntk, off, i0, ni


def walk(j, s, lq, lk, causal):
    _, _, _, i0, _ = unit_geometry(j, lq, lk, causal)
    return i0 + s if causal else s


def rank(j, i, lq, lk, causal):
    nt, ntk, off, _, _ = unit_geometry(j, lq, lk, causal)
    jmax = min(ntk - 1, floor_div((i + 1) * TILE + off - 1, TILE)) if causal else ntk - 1
    return jmax - j


def check(lq_list, lk_list, H, causal, run=1):
    """H query heads in runs of `run` heads per unit (heads of one run walked
    one after the other)."""
    assert H % run == 0
    order = unit_order(lk_list, H // run)
    pos = {u: p for p, u in enumerate(order)}
    contributions = {}  # (b, h, i) -> [(rank, position, j)]
    for (b, j, u), p in pos.items():
        lq, lk = lq_list[b], lk_list[b]
        _, _, _, _, ni = unit_geometry(j, lq, lk, causal)
        for h in range(u * run, (u + 1) * run):
            for s in range(ni):
                i = walk(j, s, lq, lk, causal)
                contributions.setdefault((b, h, i), []).append(
                    (rank(j, i, lq, lk, causal), p, j))
    for key, cs in contributions.items():
        ranks = sorted(r for r, _, _ in cs)
        assert ranks == list(range(len(cs))), (key, ranks)
        by_rank = sorted(cs)
        for (r0, p0, j0), (r1, p1, j1) in zip(by_rank, by_rank[1:]):
            assert p0 < p1, (key, "rank", r0, "unit j", j0, "taken after rank", r1, "unit j", j1)
    # every query tile of every sequence with keys receives every key/value
    # tile that some row of it sees
    for b, (lq, lk) in enumerate(zip(lq_list, lk_list)):
        for i in range(cdiv(lq, TILE)):
            rows = range(i * TILE, min((i + 1) * TILE, lq))
            want = set()
            for r in rows:
                last = min(lk - 1, r + lk - lq) if causal else lk - 1
                want.update(range(0, last // TILE + 1) if last >= 0 else [])
            got = {j for _, _, j in contributions.get((b, 0, i), [])}
            assert got == want, (b, i, sorted(want), sorted(got))


@pytest.mark.parametrize("run", [1, 2, 4])
@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths(causal, run):
    for lengths in ([2048] * 4, [1, 127, 128, 129, 300, 4097], [32768]):
        check(lengths, lengths, 4, causal, run)


@pytest.mark.parametrize("causal", [False, True])
def test_different_lengths(causal):
    cases = [([2048] * 2, [8192] * 2), ([300, 200, 129], [129, 64, 1]),
             ([129, 1, 300, 77], [400, 513, 300, 1000]), ([100, 60], [300, 60]),
             ([0, 50, 128], [200, 0, 128])]
    for lq, lk in cases:
        check(lq, lk, 2, causal)
        check(lq, lk, 4, causal, run=2)


def test_random_geometries():
    rng = random.Random(5)
    for _ in range(200):
        B = rng.randint(1, 6)
        lq = [rng.randint(0, 1500) for _ in range(B)]
        lk = [rng.choice([q, rng.randint(0, 3000)]) for q in lq]
        for causal in (False, True):
            check(lq, lk, 2, causal)
