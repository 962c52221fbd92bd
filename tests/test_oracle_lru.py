"""Pins for the oracle's literal LRU list (CPU only).

The oracle keeps the explainer page's doubly linked list. It is checked
against an independent formulation written here (each slot carries the clock
value of its last use; a miss takes the slot with the smallest value), over
every short trace of a tiny cache and over long random traces, plus the
invariants the page states and the toy hit-rate table it prints.
"""
import itertools
import os
import random

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


class ClockLRU:
    """Same transaction as the page, restated with last-use clock values."""

    def __init__(self, L, E, shared, K, max_cache_tokens=32):
        self.L, self.E, self.shared, self.K, self.mct = L, E, shared, K, max_cache_tokens
        npools = 1 if shared else L
        # slot s starts with clock s - K: slot 0 is the least recently used
        self.last = [[s - K for s in range(K)] for _ in range(npools)]
        self.owner = [[None] * K for _ in range(npools)]
        self.where = {}  # (layer, e) -> slot
        self.clock = 0

    def call(self, layer, ids, T=1):
        pool = 0 if self.shared else layer
        uniq = list(dict.fromkeys(int(i) for i in ids))
        resident = {e for e in uniq if (layer, e) in self.where}
        if T > self.mct:
            return [self.where.get((layer, int(i)), -1) for i in ids], [int(i) in resident for i in ids], []
        if len(uniq) > self.K:
            raise oracle.CacheError(oracle.ERR_CAPACITY)
        for e in uniq:
            if e in resident:
                self.last[pool][self.where[(layer, e)]] = self.clock
                self.clock += 1
        fills = []
        for e in sorted(set(uniq) - resident):
            s = min(range(self.K), key=lambda j: self.last[pool][j])
            if self.owner[pool][s] is not None:
                del self.where[self.owner[pool][s]]
            self.owner[pool][s] = (layer, e)
            self.where[(layer, e)] = s
            self.last[pool][s] = self.clock
            self.clock += 1
            fills.append((e, s))
        return [self.where[(layer, int(i))] for i in ids], [int(i) in resident for i in ids], fills

    def order(self, pool):
        return sorted(range(self.K), key=lambda j: self.last[pool][j])


def _check_same(c, m, layer, ids, T=1):
    try:
        r = c.plan(layer, ids, T)
    except oracle.CacheError as ex:
        with pytest.raises(oracle.CacheError):
            m.call(layer, ids, T)
        return ex
    so, hit, fills = m.call(layer, ids, T)
    assert list(r["slot_of"]) == so
    assert [bool(h) for h in r["hit_of"]] == hit
    assert list(zip(r["fill_expert"], r["fill_slot"])) == fills
    st = c.state()
    for p in range(c.n_pools):
        assert list(st["order"][p]) == m.order(p)
    return r


def test_exhaustive_tiny_traces_match_clock_model():
    E = 4
    calls = [list(c) for n in (1, 2, 3) for c in itertools.product(range(E), repeat=n)]
    for K in (1, 2, 3):
        for seq in itertools.product(calls, repeat=2):
            c = oracle.Cache(1, E, "per_layer", K)
            m = ClockLRU(1, E, False, K)
            for ids in seq:
                _check_same(c, m, 0, ids)
    # a denser sweep of three-call traces at K = 2
    short = [list(c) for n in (1, 2) for c in itertools.product(range(E), repeat=n)]
    for seq in itertools.product(short, repeat=3):
        c = oracle.Cache(1, E, "per_layer", 2)
        m = ClockLRU(1, E, False, 2)
        for ids in seq:
            _check_same(c, m, 0, ids)


@pytest.mark.parametrize("shared", [False, True])
def test_long_random_traces_match_clock_model(shared):
    rng = random.Random(7)
    L, E, K, k = 3, 24, 9, 3
    c = oracle.Cache(L, E, "shared" if shared else "per_layer", K)
    m = ClockLRU(L, E, shared, K)
    for step in range(1500):
        layer = rng.randrange(L)
        T = rng.choice([1, 1, 2, 3, 40])
        ids = []
        for _ in range(T):
            ids += rng.sample(range(E), k) if rng.random() < 0.5 else rng.sample(range(6), k)
        _check_same(c, m, layer, ids, T)


def test_invariants_hold_on_every_call():
    rng = random.Random(3)
    L, E, K = 2, 30, 12
    c = oracle.Cache(L, E, "shared", K, slot_bytes=100.0)
    for step in range(600):
        layer = rng.randrange(L)
        ids = [rng.randrange(E) for _ in range(rng.choice([2, 4, 8, 12]))]
        before = c.state()
        r = c.plan(layer, ids, T=len(ids))
        st = c.state()
        sm, ko = st["slot_map"], st["key_of"][0]
        # slot_map and key_of are mutual inverses
        for s, key in enumerate(ko):
            if key >= 0:
                assert sm[key // E, key % E] == s
        for l in range(L):
            for e in range(E):
                if sm[l, e] >= 0:
                    assert ko[sm[l, e]] == l * E + e
        # hits + misses = unique experts of the call
        assert r["n_hit"] + r["n_fill"] == r["n_uniq"] == len(set(ids))
        # no victim held an expert of this call
        for s in r["fill_slot"]:
            old = before["key_of"][0][s]
            assert old < 0 or not (old // E == layer and old % E in set(ids))
        # every id resolves to a slot holding it
        for i, e in enumerate(ids):
            assert ko[r["slot_of"][i]] == layer * E + e
        # the list is a permutation of the slots
        assert sorted(st["order"][0]) == list(range(K))


def test_capacity_error_leaves_state_untouched():
    c = oracle.Cache(1, 16, "per_layer", 4)
    c.plan(0, [1, 2, 3])
    before = c.state()
    with pytest.raises(oracle.CacheError) as ei:
        c.plan(0, [5, 6, 7, 8, 9])
    assert ei.value.code == oracle.ERR_CAPACITY
    after = c.state()
    for key in before:
        assert np.array_equal(before[key], after[key])
    # exactly K distinct is accepted (tokens*k = K is the edge of the rule)
    c.plan(0, [5, 6, 7, 8, 5, 6])


def test_all_resident_when_pool_holds_everything():
    L, E = 3, 10
    c = oracle.Cache(L, E, "shared", L * E)
    rng = random.Random(1)
    seen = set()
    misses = 0
    for _ in range(300):
        layer = rng.randrange(L)
        ids = rng.sample(range(E), 4)
        r = c.plan(layer, ids)
        misses += r["n_fill"]
        seen |= {(layer, e) for e in ids}
    assert misses == len(seen)  # no eviction ever: every key misses once


def test_prefill_lookup_does_not_touch_the_list():
    c = oracle.Cache(2, 20, "per_layer", 6, max_cache_tokens=32)
    c.plan(0, [1, 2, 3, 4])
    before = c.state()
    ids = list(range(20)) * 3
    r = c.plan(0, ids, T=60)
    after = c.state()
    for key in before:
        assert np.array_equal(before[key], after[key])
    assert r["n_hit"] == 4 and r["n_fill"] == 0 and r["n_uniq"] == 20
    assert all(r["slot_of"][i] == -1 for i, e in enumerate(ids) if e not in (1, 2, 3, 4))
    s = c.stats()
    assert s[2] == {"calls": 1, "hits": 4, "misses": 16, "bytes": 0}


def test_sorted_misses_into_an_empty_pool_merge_into_one_copy():
    c = oracle.Cache(1, 64, "per_layer", 16)
    r = c.plan(0, [9, 3, 7, 4, 5, 8, 6])
    assert list(r["fill_expert"]) == [3, 4, 5, 6, 7, 8, 9]
    assert list(r["fill_slot"]) == [0, 1, 2, 3, 4, 5, 6]
    assert oracle.count_runs(r["fill_expert"], r["fill_slot"]) == 1
    assert oracle.count_runs([1, 2, 5], [0, 1, 2]) == 2
    assert oracle.count_runs([], []) == 0


def test_hits_are_touched_before_any_eviction():
    # K = 2: slot 0 holds 1, slot 1 holds 2, 1 is least recent. A call with
    # [3, 1]: 1 is touched first, so 3 evicts 2 (not 1).
    c = oracle.Cache(1, 8, "per_layer", 2)
    c.plan(0, [1])
    c.plan(0, [2])
    r = c.plan(0, [3, 1])
    st = c.state()
    assert st["slot_map"][0, 1] == 0 and st["slot_map"][0, 2] == -1 and st["slot_map"][0, 3] == 1
    assert list(r["hit_of"]) == [0, 1]


def test_stats_buckets_by_batch_size():
    c = oracle.Cache(1, 64, "per_layer", 40, slot_bytes=10.0)
    c.plan(0, list(range(8)), T=8)
    c.plan(0, list(range(4, 20)), T=9)
    c.plan(0, list(range(64)), T=33)
    s = c.stats()
    assert s[0] == {"calls": 1, "hits": 0, "misses": 8, "bytes": 80}
    assert s[1] == {"calls": 1, "hits": 4, "misses": 12, "bytes": 120}
    assert s[2]["calls"] == 1 and s[2]["hits"] == 20 and s[2]["misses"] == 44


def _toy_trace(E, k, stick, tokens, seed):
    """The explainer's toy router: each token draws k distinct experts; each
    draw repeats one of the previous token's experts with probability stick,
    otherwise it takes floor(U^1.8 * E) (low ids are popular)."""
    rnd = random.Random(seed)
    prev, trace = [], []
    for _ in range(tokens):
        chosen = []
        while len(chosen) < k:
            if prev and rnd.random() < stick:
                e = prev[rnd.randrange(len(prev))]
            else:
                e = min(E - 1, int(rnd.random() ** 1.8 * E))
            if e not in chosen:
                chosen.append(e)
        prev = sorted(chosen)
        trace.append(prev)
    return trace


def test_toy_hit_rate_table_within_three_points():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "toy_lru_table.txt")) if l.strip() and l[0] != "#"]
    for stick, slots, hit_pct, upl in rows:
        stick, slots, hit_pct, upl = float(stick), int(slots), float(hit_pct), float(upl)
        hits = misses = 0
        for seed in (11, 12):
            trace = _toy_trace(512, 10, stick, 4000, seed)
            c = oracle.Cache(1, 512, "per_layer", slots)
            for picks in trace:
                r = c.plan(0, picks)
                hits += r["n_hit"]
                misses += r["n_fill"]
        ours = 100.0 * hits / (hits + misses)
        assert abs(ours - hit_pct) <= 3.0, (stick, slots, ours, hit_pct)
        assert abs(misses / 8000 - upl) <= 0.3, (stick, slots, misses / 8000, upl)
