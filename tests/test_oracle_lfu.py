"""Pins for the oracle's LFU eviction policy (CPU only).

The explainer page prints an LFU column beside its toy LRU replay, and the
FP4 page evicts the least frequently used expert; neither prints the rule.
The oracle's reading: every key counts the calls that routed it over the
whole history, and a miss takes, among the slots its call does not hold, the
one whose key has the fewest uses (empty slots first), least recently used
on ties. Checked against the toy table's LFU column, a worked example where
LRU and LFU part, and an LFU restated here over random traces.
"""
import os
import random

import numpy as np
import pytest

import oracle
from test_oracle_lru import _toy_trace

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


class CountLFU:
    """The same reading restated: per-key use counts, a recency list per pool."""

    def __init__(self, L, E, shared, K):
        self.E, self.shared, self.K = E, shared, K
        npools = 1 if shared else L
        self.order = [list(range(K)) for _ in range(npools)]  # least recent first
        self.owner = [[None] * K for _ in range(npools)]
        self.where = {}
        self.uses = {}

    def call(self, layer, ids, T=1):
        pool = 0 if self.shared else layer
        uniq = list(dict.fromkeys(int(i) for i in ids))
        if len(uniq) > self.K:
            raise oracle.CacheError(oracle.ERR_CAPACITY)
        for e in uniq:
            self.uses[(layer, e)] = self.uses.get((layer, e), 0) + 1
        resident = {e for e in uniq if (layer, e) in self.where}
        held = set()
        for e in uniq:
            if e in resident:
                s = self.where[(layer, e)]
                self.order[pool].remove(s)
                self.order[pool].append(s)
                held.add(s)
        fills = []
        for e in sorted(set(uniq) - resident):
            cand = [s for s in self.order[pool] if s not in held]
            s = min(cand, key=lambda q: (-1 if self.owner[pool][q] is None else self.uses[self.owner[pool][q]],
                                         self.order[pool].index(q)))
            if self.owner[pool][s] is not None:
                del self.where[self.owner[pool][s]]
            self.owner[pool][s] = (layer, e)
            self.where[(layer, e)] = s
            self.order[pool].remove(s)
            self.order[pool].append(s)
            held.add(s)
            fills.append((e, s))
        return [self.where[(layer, int(i))] for i in ids], [int(i) in resident for i in ids], fills


def test_lfu_and_lru_part_where_the_frequent_expert_is_the_least_recent():
    # two slots; expert 0 twice, then 1, then 2: LRU evicts 0 (least recent),
    # LFU evicts 1 (used once against 0's twice)
    lfu = oracle.Cache(1, 4, "per_layer", 2, policy="lfu")
    lru = oracle.Cache(1, 4, "per_layer", 2)
    for ids in ([0], [0], [1]):
        lfu.plan(0, ids)
        lru.plan(0, ids)
    a, b = lfu.plan(0, [2]), lru.plan(0, [2])
    assert list(a["fill_slot"]) == [1] and list(b["fill_slot"]) == [0]
    assert list(lfu.state()["slot_map"][0]) == [0, -1, 1, -1]
    assert list(lru.state()["slot_map"][0]) == [-1, 1, 0, -1]


def test_an_invalid_policy_is_refused():
    with pytest.raises(ValueError):
        oracle.Cache(1, 4, "per_layer", 2, policy="mru")


@pytest.mark.parametrize("shared", [False, True])
def test_lfu_matches_the_restated_policy_on_random_traces(shared):
    rng = random.Random(23 + shared)
    for trial in range(30):
        L, E, k = 3, rng.choice([8, 12, 16]), rng.choice([2, 3])
        K = rng.randint(k * 2, 3 * k + 4)
        ref = oracle.Cache(L, E, "shared" if shared else "per_layer", K, policy="lfu")
        alt = CountLFU(L, E, shared, K)
        for step in range(60):
            T = rng.randint(1, 2)
            layer = rng.randrange(L)
            ids = np.array([rng.sample(range(E), k) for _ in range(T)], dtype=np.int32).reshape(-1)
            p = ref.plan(layer, ids, T)
            slots, hits, fills = alt.call(layer, ids, T)
            assert list(p["slot_of"]) == slots
            assert [bool(h) for h in p["hit_of"]] == hits
            assert list(zip(p["fill_expert"], p["fill_slot"])) == fills


def test_lfu_never_evicts_an_expert_of_the_same_call_and_equals_lru_without_evictions():
    rng = random.Random(5)
    E, k = 16, 4
    for K in (4, 6, 16):
        lfu = oracle.Cache(1, E, "per_layer", K, policy="lfu")
        lru = oracle.Cache(1, E, "per_layer", K)
        for step in range(200):
            ids = np.array(rng.sample(range(E), k), dtype=np.int32)
            a, b = lfu.plan(0, ids), lru.plan(0, ids)
            # every pick ends resident in a distinct slot
            assert len(set(a["slot_of"].tolist())) == k and (a["slot_of"] >= 0).all()
            if K == E:
                assert np.array_equal(a["slot_of"], b["slot_of"])


def test_toy_lfu_column():
    # Without locality (stickiness 0) the toy's LFU column is the hit rate of
    # the most used experts, and this policy lands within three points of it.
    # With locality the toy's LFU barely gains (18-19% at 25 slots): its
    # replay admits one pick at a time, so a token's new experts evict each
    # other before the next token can reuse them. A cache call holds all of
    # its experts (none can evict another), so here locality does pay, and
    # the hit rate is at least the page's.
    rows = [l.split() for l in open(os.path.join(GOLDEN, "toy_lfu_table.txt")) if l.strip() and l[0] != "#"]
    for stick, slots, hit_pct, upl in rows:
        stick, slots, hit_pct, upl = float(stick), int(slots), float(hit_pct), float(upl)
        hits = misses = 0
        for seed in (11, 12):
            trace = _toy_trace(512, 10, stick, 4000, seed)
            c = oracle.Cache(1, 512, "per_layer", slots, policy="lfu")
            for picks in trace:
                r = c.plan(0, picks)
                hits += r["n_hit"]
                misses += r["n_fill"]
        ours = 100.0 * hits / (hits + misses)
        if stick == 0.0:
            assert abs(ours - hit_pct) <= 3.0, (stick, slots, ours, hit_pct)
            assert abs(misses / 8000 - upl) <= 0.3, (stick, slots, misses / 8000, upl)
        else:
            assert ours >= hit_pct - 3.0, (stick, slots, ours, hit_pct)
