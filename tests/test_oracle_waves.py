"""Pins for the oracle's wave split of a decode step (CPU only).

[PAGED, "What happens with more than one request?"]: a step is one wave only
if tokens x top_k <= K, so up to K // top_k tokens; larger steps run several
waves, each with its own page-in. The oracle groups tokens in order, K // top_k
per wave. Checked against the page's table of K // 8, the single-wave rule,
and a brute-force replay of the waves through an independent LRU.
"""
import os
import random

import numpy as np
import pytest

import oracle
from test_oracle_lru import ClockLRU

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "waves_paged.txt")


def _table():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        name, K, per, wins = line.split()
        rows.append((name, int(K), int(per), wins == "yes"))
    return rows


@pytest.mark.parametrize("name,K,per,wins", _table())
def test_page_table_single_wave_batch(name, K, per, wins):
    # K // 8 on the page is the largest batch the oracle serves in one wave
    assert oracle.wave_split(per, 8, K) == [(0, per)]
    assert len(oracle.wave_split(per + 1, 8, K)) == 2
    # four requests: one wave exactly on the runs the page says win
    assert (len(oracle.wave_split(4, 8, K)) == 1) == wins


@pytest.mark.parametrize("T,k,K", [(1, 1, 1), (5, 8, 12), (7, 4, 10), (32, 8, 92), (32, 10, 31), (13, 3, 40),
                                   (32, 16, 16), (9, 2, 17)])
def test_waves_cover_the_tokens_in_order_within_the_rule(T, k, K):
    waves = oracle.wave_split(T, k, K)
    per = K // k
    assert len(waves) == -(-T // per)
    t = 0
    for i, (s, n) in enumerate(waves):
        assert s == t and 1 <= n and n * k <= K
        if i < len(waves) - 1:
            assert n == per
        t += n
    assert t == T
    if T * k <= K:
        assert waves == [(0, T)]


def test_no_wave_fits_when_the_pool_is_smaller_than_top_k():
    assert oracle.wave_split(3, 8, 7) == []


def test_wave_replay_matches_an_independent_lru():
    # The waves of each step go through the literal list one after another;
    # the clock-value LRU written in this file, fed the same waves, gives the
    # same slots, hits and fills, and no wave exceeds the pool.
    rng = random.Random(7)
    for trial in range(40):
        L, E, k = 2, rng.choice([8, 16, 24]), rng.choice([2, 3, 4])
        K = rng.randint(k, 2 * k + 3)
        ref = oracle.Cache(L, E, "per_layer", K)
        alt = ClockLRU(L, E, False, K)
        for step in range(12):
            T = rng.randint(1, 8)
            layer = rng.randrange(L)
            ids = np.array([rng.sample(range(E), k) for _ in range(T)], dtype=np.int32)
            for s, n in oracle.wave_split(T, k, K):
                w_ids = ids[s:s + n].reshape(-1)
                p = ref.plan(layer, w_ids, n)
                slots, hits, fills = alt.call(layer, w_ids, n)
                assert list(p["slot_of"]) == slots
                assert [bool(h) for h in p["hit_of"]] == hits
                assert list(zip(p["fill_expert"], p["fill_slot"])) == fills
