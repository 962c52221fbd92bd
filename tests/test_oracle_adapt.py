"""Pins for the oracle's adaptive per-layer capacity (CPU only).

[FP4LOCAL] "Running a 95 GiB MoE Model on a 32 GiB GPU", "Decode": the buffer
pool is partitioned by layer, and as decoding progresses some capacity is
moved from layers with high hit rates to layers with low hit rates, with the
same total. The page prints no rule; the oracle's reading (every period * L
decode calls, `step` slots move from the highest to the lowest window hit
rate, within [kmin, kmax]; a moved slot leaves as the giver's least recently
used and arrives as the taker's empty least recently used) is pinned by:
- a worked example computed by hand below;
- the invariants: total capacity constant, the bounds held, every list as
  long as its pool, the slot map and the keys mutual inverses;
- an independent restatement written here (last-use clock values and
  dictionaries, rates compared as fractions) over random traces.
"""
import random
from fractions import Fraction

import numpy as np
import pytest

import oracle


def test_worked_example():
    # 3 layers of 3 slots, top-1, a move every 3 decode calls (period 1)
    c = oracle.Cache(3, 8, "per_layer", 3, slot_bytes=1.0, adaptive=(1, 1, 2, 5))
    one = lambda l, e: c.plan(l, np.array([e], dtype=np.int32), 1)
    # window 1: every layer misses once -> equal rates -> no move
    for l in range(3):
        assert one(l, 1)["fill_slot"].tolist() == [0]
    assert c.pool_slots() == [3, 3, 3]
    # window 2: layer 0 hits (rate 1), layers 1 and 2 miss (rate 0):
    # layer 0 gives its least recently used slot (slot 1, still empty) to
    # layer 1 (the lowest rate, lower layer first), where it becomes place 3
    assert one(0, 1)["n_hit"] == 1
    assert one(1, 2)["fill_slot"].tolist() == [1]
    assert one(2, 3)["fill_slot"].tolist() == [1]
    assert c.pool_slots() == [2, 4, 3]
    st = c.state()
    assert st["order"][0].tolist() == [2, 0, -1, -1, -1]
    assert st["order"][1].tolist() == [3, 2, 0, 1, -1]
    assert st["key_of"][0].tolist()[:3] == [0 * 8 + 1, -1, -1]
    # the new slot is layer 1's least recently used: its next miss takes it
    assert one(1, 5)["fill_slot"].tolist() == [3]


class ClockAdaptive:
    """Per-layer pools as {place: [key, stamp]}; a miss takes the smallest stamp."""

    def __init__(self, L, K0, period, step, kmin, kmax):
        self.L, self.period, self.step, self.kmin, self.kmax = L, period, step, kmin, kmax
        self.pools = [{s: [None, s - K0] for s in range(K0)} for _ in range(L)]
        self.where = {}
        self.clock = 0
        self.low = -K0  # stamps of arriving slots go below every other
        self.calls = 0
        self.win = [[0, 0] for _ in range(L)]

    def call(self, layer, ids, T):
        pool = self.pools[layer]
        uniq = list(dict.fromkeys(int(i) for i in ids))
        if len(uniq) > len(pool):
            raise oracle.CacheError(oracle.ERR_CAPACITY)
        res = {e for e in uniq if (layer, e) in self.where}
        for e in uniq:
            if e in res:
                pool[self.where[(layer, e)]][1] = self.clock
                self.clock += 1
        fills = []
        for e in sorted(set(uniq) - res):
            s = min(pool, key=lambda p: pool[p][1])
            if pool[s][0] is not None:
                del self.where[pool[s][0]]
            pool[s] = [(layer, e), self.clock]
            self.where[(layer, e)] = s
            self.clock += 1
            fills.append((e, s))
        self.win[layer][0] += len(res)
        self.win[layer][1] += len(fills)
        self.calls += 1
        if self.calls % (self.period * self.L) == 0:
            self.rebalance()
        return [self.where[(layer, int(i))] for i in ids], fills

    def rebalance(self):
        rate = {l: Fraction(h, h + m) for l, (h, m) in enumerate(self.win) if h + m}
        give = [l for l in rate if len(self.pools[l]) - self.step >= self.kmin]
        take = [l for l in rate if len(self.pools[l]) + self.step <= self.kmax]
        if give and take:
            d = max(give, key=lambda l: (rate[l], -l))
            r = min(take, key=lambda l: (rate[l], l))
            if d != r and rate[d] > rate[r]:
                for _ in range(self.step):
                    s = min(self.pools[d], key=lambda p: self.pools[d][p][1])
                    key, _ = self.pools[d].pop(s)
                    if key is not None:
                        del self.where[key]
                    t = min(set(range(self.kmax)) - set(self.pools[r]))
                    self.low -= 1
                    self.pools[r][t] = [None, self.low]
        self.win = [[0, 0] for _ in range(self.L)]

    def order(self, layer):
        p = self.pools[layer]
        return sorted(p, key=lambda s: p[s][1]) + [-1] * (self.kmax - len(p))


@pytest.mark.parametrize("seed", range(10))
def test_random_traces_match_the_clock_restatement(seed):
    rng = random.Random(100 + seed)
    L, E, K0, k = rng.choice([(3, 12, 5, 2), (4, 16, 6, 2), (2, 10, 4, 1), (5, 20, 8, 3)])
    period, step = rng.choice([1, 2, 3]), rng.choice([1, 2])
    kmin, kmax = max(k, K0 // 2), K0 + K0 // 2 + 1
    c = oracle.Cache(L, E, "per_layer", K0, slot_bytes=1.0, adaptive=(period, step, kmin, kmax))
    m = ClockAdaptive(L, K0, period, step, kmin, kmax)
    hot = {l: rng.sample(range(E), rng.randint(2, E)) for l in range(L)}  # layers differ in locality
    for _ in range(300):
        layer = rng.randrange(L)
        T = rng.randint(1, max(1, kmin // k))
        ids = [rng.choice(hot[layer]) for _ in range(T * k)]
        so, fills = m.call(layer, ids, T)
        r = c.plan(layer, np.array(ids, dtype=np.int32), T)
        assert list(r["slot_of"]) == so
        assert list(zip(r["fill_expert"], r["fill_slot"])) == fills
        assert c.pool_slots() == [len(p) for p in m.pools]
    st = c.state()
    for l in range(L):
        assert st["order"][l].tolist() == m.order(l)


@pytest.mark.parametrize("seed", range(6))
def test_invariants(seed):
    rng = random.Random(seed)
    L, E, K0, k = 4, 24, 8, 2
    c = oracle.Cache(L, E, "per_layer", K0, slot_bytes=1.0, adaptive=(2, 1, 4, 12))
    for _ in range(400):
        layer = rng.randrange(L)
        span = 3 + 5 * layer  # layer 0 reuses few experts, layer 3 many
        ids = np.array([rng.randrange(span) for _ in range(k)], dtype=np.int32)
        c.plan(layer, ids, 1)
        sizes = c.pool_slots()
        assert sum(sizes) == L * K0 and all(4 <= s <= 12 for s in sizes)
    st = c.state()
    sizes = c.pool_slots()
    for l in range(L):
        order = st["order"][l].tolist()
        assert all(s >= 0 for s in order[:sizes[l]]) and all(s == -1 for s in order[sizes[l]:])
        for e in range(E):
            s = st["slot_map"][l][e]
            if s >= 0:
                assert st["key_of"][l][s] == l * E + e and s in order[:sizes[l]]
    assert sizes[3] > sizes[0]  # capacity went to the layer that misses more


def test_adaptive_needs_per_layer_pools_and_sane_bounds():
    with pytest.raises(ValueError):
        oracle.Cache(2, 16, "shared", 8, adaptive=(1, 1, 4, 12))
    with pytest.raises(ValueError):
        oracle.Cache(2, 16, "per_layer", 8, adaptive=(1, 1, 9, 12))
