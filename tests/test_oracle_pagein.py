"""Pins for the oracle's page-in prefill (CPU only).

[PAGED] "Running an MoE Model Larger Than Your VRAM: SGLang Paged Experts, the
PCIe Math, and the 4-Request Cliff", "Why do short prompts get slower first
tokens?": a prefill touches nearly every expert, so it pages in everything
that is not resident, once. The oracle reads this as the decode transaction
over all of the call's distinct experts, without the capacity rule. Pinned by:
- the page's three worked page-in volumes (K = 92, 40 and 26 of 128 experts);
- an independent formulation written here (last-use clock values; a miss
  takes the slot with the smallest value, whoever touched it) over random
  traces that mix decode calls and prefills with more distinct experts than
  slots;
- the invariants the page implies (every routed expert resident afterwards
  when they fit; the read-only prefill leaves the list alone).
"""
import os
import random

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_arithmetic.txt")


def golden(name):
    for line in open(GOLDEN):
        f = line.split()
        if f and not line.startswith("#") and f[0] == name:
            return float(f[1])
    raise KeyError(name)


@pytest.mark.parametrize("K,expert_mb,volume", [(92, "paged_int4_expert_MB", "paged_int4_pagein_GB"),
                                                (40, "paged_fp8_expert_MB", "paged_fp8_pagein_GB"),
                                                (26, "paged_int4_expert_MB", "paged_laptop_pagein_GB")])
def test_page_in_volume_matches_the_page(K, expert_mb, volume):
    # Qwen3-30B-A3B: 48 layers of 128 experts, top-8. A "slot" on the page is
    # one expert of every layer (48 x 2.43 MB int4, 48 x 4.72 MB FP8; printed
    # rounded as 117 and 227 MB), so one layer's pool with that many bytes
    # per slot counts what all 48 layers move. Decode fills the K slots; a
    # prefill that routes all 128 experts then pages in the other 128 - K,
    # once each, even where 128 > K. The page's volumes are "about" values.
    E = 128
    c = oracle.Cache(1, E, "per_layer", K, slot_bytes=48 * golden(expert_mb) * 1e6, prefill="page_in")
    for i in range(0, K, 8):
        c.plan(0, np.arange(i, min(i + 8, K), dtype=np.int32), 1)
    before = c.stats()[2]["bytes"]
    ids = np.resize(np.arange(E, dtype=np.int32)[::-1], 33 * 8)  # a 33-token prefill over every expert
    r = c.plan(0, ids, 33)
    assert r["n_hit"] == K and r["n_fill"] == E - K
    moved = c.stats()[2]["bytes"] - before
    assert abs(moved / 1e9 - golden(volume)) < 0.05, moved / 1e9


class ClockPageIn:
    """The transaction restated with last-use clock values (one pool)."""

    def __init__(self, E, K, mct=32, page_in=True):
        self.E, self.K, self.mct, self.page_in = E, K, mct, page_in
        self.last = [s - K for s in range(K)]
        self.owner = [None] * K
        self.where = {}
        self.clock = 0

    def call(self, ids, T):
        uniq = list(dict.fromkeys(int(i) for i in ids))
        resident = {e for e in uniq if e in self.where}
        if T > self.mct and not self.page_in:
            return [self.where.get(int(i), -1) for i in ids], [int(i) in resident for i in ids], []
        if T <= self.mct and len(uniq) > self.K:
            raise oracle.CacheError(oracle.ERR_CAPACITY)
        used = {}
        for e in uniq:
            if e in resident:
                used[e] = self.where[e]
                self.last[used[e]] = self.clock
                self.clock += 1
        fills = []
        for e in sorted(set(uniq) - resident):
            s = min(range(self.K), key=lambda j: self.last[j])
            if self.owner[s] is not None:
                del self.where[self.owner[s]]
            self.owner[s] = e
            self.where[e] = s
            used[e] = s
            self.last[s] = self.clock
            self.clock += 1
            fills.append((e, s))
        return [used[int(i)] for i in ids], [int(i) in resident for i in ids], fills

    def order(self):
        return sorted(range(self.K), key=lambda j: self.last[j])


@pytest.mark.parametrize("seed", range(12))
def test_random_traces_match_the_clock_formulation(seed):
    rng = random.Random(seed)
    E, K, k = rng.choice([(12, 5, 2), (16, 6, 3), (20, 9, 2), (32, 7, 4)])
    c = oracle.Cache(1, E, "per_layer", K, slot_bytes=1.0, prefill="page_in")
    m = ClockPageIn(E, K)
    for _ in range(60):
        if rng.random() < 0.3:
            T = rng.randint(33, 40)  # a prefill, often with more distinct experts than slots
            ids = [rng.randrange(E) for _ in range(T * k)]
        else:
            T = rng.randint(1, max(1, K // k))
            ids = [rng.randrange(E) for _ in range(T * k)]
        so, hit, fills = m.call(ids, T)
        r = c.plan(0, np.array(ids, dtype=np.int32), T)
        assert list(r["slot_of"]) == so
        assert [bool(h) for h in r["hit_of"]] == hit
        assert list(zip(r["fill_expert"], r["fill_slot"])) == fills
        st = c.state()
        assert list(st["order"][0]) == m.order()
        for e in range(E):
            assert st["slot_map"][0][e] == m.where.get(e, -1)


def test_page_in_leaves_every_routed_expert_resident_when_they_fit():
    E, K = 24, 10
    c = oracle.Cache(1, E, "per_layer", K, slot_bytes=1.0, prefill="page_in")
    c.plan(0, np.array([3, 4, 5, 6], dtype=np.int32), 2)
    ids = np.array([9, 3, 11, 2, 9, 4, 15, 1] * 5, dtype=np.int32)  # 40 tokens of top-1: 7 distinct experts
    r = c.plan(0, ids, 40)
    st = c.state()
    for e in set(ids.tolist()):
        assert st["slot_map"][0][e] >= 0
    assert r["n_hit"] == 2 and r["n_fill"] == 5
    # the misses were filled ascending, so the largest one is the most recent
    assert st["order"][0][-1] == st["slot_map"][0][15]


def test_read_only_prefill_leaves_the_list_alone():
    E, K = 24, 10
    c = oracle.Cache(1, E, "per_layer", K, slot_bytes=1.0)
    c.plan(0, np.array([3, 4, 5, 6], dtype=np.int32), 2)
    before = c.state()
    r = c.plan(0, np.arange(E, dtype=np.int32), 40)
    after = c.state()
    for key in before:
        assert np.array_equal(before[key], after[key])
    assert r["n_fill"] == 0 and r["n_hit"] == 4


def test_page_in_needs_lru():
    with pytest.raises(ValueError):
        oracle.Cache(1, 16, "per_layer", 8, policy="lfu", prefill="page_in")
