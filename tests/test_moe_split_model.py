"""CPU model of the grouped decode GEMV's work split and hand-over protocol (csrc/moe.cu).

Not the CUDA code itself: a line-by-line model of its integer arithmetic and its barrier
protocol, checked over random routings and shapes --
* the cost-weighted stream-K split (share_start, the reducer's owner arithmetic): every
  share non-empty, every unit owned by the share the reducer computes, and no row tile met
  by more CTAs than the parts the host sizes the workspace for (grouped_parts);
* the producer / twelve consumer warps / reducer protocol over random schedules: no
  deadlock, no mbarrier phase lapped, every unit consumed once by its two warps into the
  piece of its row tile.
"""
import random

import pytest

KGCW = 12          # consumer warps
KGC = KGCW // 2    # units per chunk


def unit_cost(m):
    return 2 * m + 3


def grouped_parts(T, topk, nt, kg, grid):
    cmin = nt * kg * (2 * T * topk + 3 * topk)
    span = kg * unit_cost(T) * grid
    return min(kg, (span + cmin - 1) // cmin + 1)


def split(T, topk, NT, KG, grid, cnts, shared):
    """(G, share starts, C(u) per unit, cost prefix per group, unit cost per group)."""
    n_active = len(cnts)
    UG = NT * KG
    first = [sum(cnts[:g]) for g in range(n_active)]
    wmax = unit_cost(T)
    Csh = UG * (2 * T * topk + 3 * n_active)
    Ctot = Csh + (UG * wmax if shared else 0)
    G = max(1, min(grid, Ctot // wmax))
    cg = [UG * (2 * first[g] + 3 * g) for g in range(n_active)] + ([Csh] if shared else [])
    wg = [unit_cost(min(4, c)) for c in cnts] + ([wmax] if shared else [])
    n_groups = len(cg)

    def share_start(bb):
        if bb >= G:
            return n_groups * UG
        tgt = bb * Ctot
        gs = sum(1 for g in range(n_groups) if cg[g] * G <= tgt) - 1
        wG = wg[gs] * G
        j = (tgt - cg[gs] * G + wG - 1) // wG
        return min(gs * UG + j, (gs + 1) * UG)

    C = [cg[g] + l * wg[g] for g in range(n_groups) for l in range(UG)]
    return G, Ctot, [share_start(b) for b in range(G + 1)], C, cg, wg


def random_routing(rng, T, topk, E):
    counts = {}
    base = rng.sample(range(E), topk)
    same = rng.random() < 0.3
    for _ in range(T):
        for e in (base if same else rng.sample(range(E), topk)):
            counts[e] = counts.get(e, 0) + 1
    return [counts[e] for e in sorted(counts)]


@pytest.mark.parametrize("seed", range(4))
def test_weighted_split_shares_owners_and_part_bound(seed):
    rng = random.Random(seed)
    for _ in range(400):
        T, topk = rng.randint(1, 4), rng.randint(1, 16)
        E = max(topk, rng.choice([topk, 16, 64, 512]))
        cnts = random_routing(rng, T, topk, E)
        NT, KG = rng.choice([1, 2, 3, 8, 16]), rng.choice([1, 2, 4, 8, 12, 32])
        grid = rng.choice([152, 33, 7, 1])
        G, Ctot, starts, C, cg, wg = split(T, topk, NT, KG, grid, cnts, rng.random() < 0.7)
        assert C[-1] * G < (1 << 32)  # the host's 32-bit guard holds for these shapes
        for b in range(G):
            assert starts[b] < starts[b + 1]
            for u in range(starts[b], starts[b + 1]):
                assert C[u] * G // Ctot == b
        P = grouped_parts(T, topk, NT, KG, grid)
        for tile in range(len(C) // KG):
            g = tile // NT
            ct = cg[g] + (tile - g * NT) * KG * wg[g]
            assert ct == C[tile * KG]
            first_b, last_b = ct * G // Ctot, (ct + (KG - 1) * wg[g]) * G // Ctot
            assert last_b - first_b + 1 <= P


class _Bar:
    def __init__(self, count):
        self.count, self.pending, self.done = count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending, self.done = 0, self.done + 1

    def ready(self, phase):
        assert self.done <= phase + 1, "an mbarrier phase was lapped"
        return self.done > phase


def _simulate(u0, u1, NT, KG, S, rng):
    UG = NT * KG
    t0, npieces = u0 // KG, (u1 - 1) // KG - u0 // KG + 1
    chunks, c0 = [], u0
    g, gend = u0 // UG, min(u1, (u0 // UG + 1) * UG)
    while c0 < u1:
        c1 = min(c0 + KGC, gend)
        chunks.append((c0, c1, g))
        c0 = c1
        if c0 == gend:
            g, gend = g + 1, min(u1, (g + 2) * UG)
    full, empty = [_Bar(1) for _ in range(S)], [_Bar(KGCW) for _ in range(S)]
    rfull, rempty = [_Bar(KGCW) for _ in range(2)], [_Bar(1) for _ in range(2)]
    got = {}

    def producer():
        for j in range(len(chunks)):
            if j >= S:
                while not empty[j % S].ready(j // S - 1):
                    yield False
            full[j % S].arrive()
            yield True

    def flush(w, i, units):
        if i >= 2:
            while not rempty[i & 1].ready((i >> 1) - 1):
                yield False
        got.setdefault(i, []).append((w, tuple(units)))
        rfull[i & 1].arrive()
        yield True

    def consumer(w):
        ug, cur, units = w // 2, 0, []
        for j, (c0, c1, g) in enumerate(chunks):
            uw = c0 + ug
            tile = (uw if uw < c1 else c0) // KG
            while cur < tile - t0:  # every piece before this warp's unit goes first
                yield from flush(w, cur, units)
                cur, units = cur + 1, []
            while not full[j % S].ready(j // S):
                yield False
            if uw < c1:
                units.append(uw)
            empty[j % S].arrive()
            yield True
        while cur < npieces:
            yield from flush(w, cur, units)
            cur, units = cur + 1, []

    def reducer():
        for i in range(npieces):
            while not rfull[i & 1].ready(i >> 1):
                yield False
            rempty[i & 1].arrive()
            yield True

    live = [producer(), reducer()] + [consumer(w) for w in range(KGCW)]
    idle = 0
    while live:
        a = rng.choice(live)
        try:
            progressed = next(a)
        except StopIteration:
            live.remove(a)
            progressed = True
        idle = 0 if progressed else idle + 1
        assert idle < 20000, "deadlock"
    seen = set()
    for i, lst in got.items():
        assert len(lst) == KGCW
        for w, units in lst:
            for u in units:
                assert u // KG == t0 + i and (u, w % 2) not in seen
                seen.add((u, w % 2))
    assert seen == {(u, h) for u in range(u0, u1) for h in range(2)}


@pytest.mark.parametrize("seed", range(3))
def test_handover_protocol_random_schedules(seed):
    rng = random.Random(100 + seed)
    for _ in range(150):
        NT, KG = rng.choice([1, 2, 3, 8, 16]), rng.choice([1, 2, 3, 4, 8, 32])
        U = rng.randint(1, 12) * NT * KG
        u0 = rng.randrange(U)
        u1 = rng.randint(u0 + 1, min(U, u0 + rng.choice([1, 3, 7, 40, 200])))
        _simulate(u0, u1, NT, KG, rng.choice([2, 3, 4, 7]), rng)
