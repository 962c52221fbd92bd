"""Adaptive per-layer capacity ("Running a 95 GiB MoE Model on a 32 GiB GPU",
"Decode": capacity moves from layers with high hit rates to layers with low
hit rates, the total kept).

The layers route with very different locality, so slots move. Every call's
routing, slots, hits and fills, the pools' sizes after every call and the
final state must be the oracle's (its adaptive reading), on both decode
paths, with LRU and LFU eviction and with page-in prefills among the calls;
outputs stay within rel-L2 1e-3 of the oracle.
"""
import numpy as np
import pytest

import oracle
import synth
from harness import OracleRun, Setup, compare_trace, cuda_available, rel_l2
from synth.workloads import WORKLOADS, scaled

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

TOL = 1e-3


@pytest.mark.parametrize("decode,eviction,prefill", [("one_kernel", "lru", "read_only"),
                                                     ("three_kernels", "lru", "page_in"),
                                                     ("one_kernel", "lfu", "read_only"),
                                                     ("three_kernels", "lfu", "read_only")])
def test_adaptive_capacity_matches_the_oracle(decode, eviction, prefill):
    K0, adapt = 10, (2, 1, 6, 16)  # a move every 2 * L decode calls, one slot at a time
    w = scaled(WORKLOADS["qwen3_30b_a3b_q4_0"], name="adapt", L=3, E=32, k=2, H=256, I=128, slots_per_layer=K0,
               bias=True, streams=(2,), steps=40, rho=0.9)
    st = Setup(w, decode=decode, eviction=eviction, prefill=prefill, adapt=adapt, max_tokens=40)
    orc = OracleRun(w, st.info["slot_bytes"], policy=eviction, prefill=prefill, adaptive=adapt)
    # layer l's streams decorrelate faster the higher l is: the layers' hit rates differ
    xs = {l: st.hiddens(l, 2, w.steps, rho=[0.97, 0.7, 0.1][l]) for l in range(w.L)}
    moved = False
    for step in range(w.steps):
        for l in range(w.L):
            T = 1 if (step + l) % 3 else 2
            x = xs[l][step][:T]
            y = st.forward(x, l)
            ids, _ = orc.route(x, st.router[l], st.bias)
            compare_trace(st.cache.trace_read()[0], ids, orc.plan(l, ids, T), l, T)
            assert st.cache.pool_slots() == orc.cache.pool_slots()
            moved |= orc.cache.pool_slots() != [K0] * w.L
            if step % 8 == 0:
                _, _, yo = orc.layer(x, st.router[l], st.bias, l)
                assert rel_l2(y, yo) <= TOL
        if prefill == "page_in" and step % 10 == 9:
            x = synth.prompt(w.seed + step, 1, 40, w.H)
            st.forward(x, 1)
            ids, _ = orc.route(x, st.router[1], st.bias)
            compare_trace(st.cache.trace_read()[0], ids, orc.plan(1, ids, 40), 1, 40)
    assert moved
    sizes = st.cache.pool_slots()
    assert sum(sizes) == w.L * K0 and sizes[2] > sizes[0]
    g, o = st.cache.state(), orc.cache.state()
    for key in ("slot_map", "key_of", "order"):
        assert np.array_equal(g[key], o[key]), key
    for p in range(w.L):
        for s, key in enumerate(g["key_of"][p]):
            if key >= 0:
                dev, store = st.cache.read_slot(p, s, key // w.E, key % w.E)
                assert np.array_equal(dev, store)
    st.close()
