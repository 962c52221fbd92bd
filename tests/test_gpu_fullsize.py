"""Parity at the workloads' full sizes, through the same C-ABI calls bench.py
times: routing, slots, hits and fills bit-exact on every call; layer outputs
(rel-L2 <= 1e-3) on sampled calls, where the oracle evaluates the whole
unpaged layer; the final LRU order of every pool; byte-exact slot contents.
"""
import numpy as np
import pytest

import synth
from harness import OracleRun, Setup, compare_trace, cuda_available, rel_l2
from synth.workloads import WORKLOADS

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

TOL = 1e-3


def decode_run(st, orc, steps, T, sample):
    """sample: set of (step, layer) whose outputs are compared with the oracle."""
    w = st.w
    xs = {l: st.hiddens(l, T, steps) for l in range(w.L)}
    worst = 0.0
    for step in range(steps):
        for l in range(w.L):
            x = xs[l][step]
            y = st.forward(x, l)
            ids, _ = orc.route(x, st.router[l], st.bias)
            plan = orc.plan(l, ids, T)
            compare_trace(st.cache.trace_read()[0], ids, plan, l, T)
            if (step, l) in sample:
                _, _, yo = orc.layer(x, st.router[l], st.bias, l)
                err = rel_l2(y, yo)
                worst = max(worst, err)
                assert err <= TOL, (step, l, err)
    return worst


def check_state(st, orc, spot_slots=4):
    g, o = st.cache.state(), orc.cache.state()
    assert np.array_equal(g["slot_map"], o["slot_map"])
    assert np.array_equal(g["key_of"], o["key_of"])
    assert np.array_equal(g["order"], o["order"])
    E = st.w.E
    checked = 0
    for p in range(g["key_of"].shape[0]):
        for s in range(g["key_of"].shape[1] - 1, -1, -1):
            key = int(g["key_of"][p, s])
            if key >= 0:
                dev, store = st.cache.read_slot(p, s, key // E, key % E)
                assert np.array_equal(dev, store), (p, s, key)
                checked += 1
                break
        if checked >= spot_slots:
            break


def test_qwen3_30b_a3b_q4_0_full():
    w = WORKLOADS["qwen3_30b_a3b_q4_0"]
    st = Setup(w)
    orc = OracleRun(w, st.info["slot_bytes"])
    steps = 24
    worst = decode_run(st, orc, steps, 1, {(s, l) for s in (0, 12, 23) for l in (0, 23, 47)})
    check_state(st, orc)
    print("q4_0 full: worst rel-L2", worst, st.cache.stats()["buckets"][0])
    st.close()


def test_qwen3_30b_a3b_fp8_full_batch8():
    w = WORKLOADS["qwen3_30b_a3b_fp8"]
    st = Setup(w, max_tokens=8)
    orc = OracleRun(w, st.info["slot_bytes"])
    worst = decode_run(st, orc, 6, 8, {(s, l) for s in (0, 5) for l in (0, 47)})
    check_state(st, orc)
    print("fp8 full T=8: worst rel-L2", worst)
    st.close()


def test_flash_next_nvfp4_shared_pool_full():
    w = WORKLOADS["flash_next_nvfp4"]
    st = Setup(w)
    assert st.info["slots_per_pool"] == 4031 and st.info["num_pools"] == 1
    orc = OracleRun(w, st.info["slot_bytes"])
    # 40 steps x 48 layers fill the 4031-slot pool and evict across layers
    worst = decode_run(st, orc, 40, 1, {(s, l) for s in (0, 39) for l in (0, 31)})
    check_state(st, orc)
    s = st.cache.stats()["buckets"][0]
    assert s["misses"] > 4031  # evictions happened
    print("nvfp4 shared pool full: worst rel-L2", worst, s)
    st.close()


def test_flash_next_prefill_and_batch32_full():
    w = WORKLOADS["flash_next_prefill"]
    st = Setup(w, max_tokens=w.prompt_T)
    orc = OracleRun(w, st.info["slot_bytes"])
    # fill the pool with decode batches of 32, then prefill two layers
    decode_run(st, orc, 2, 32, {(1, 0)})
    before = st.cache.state()
    for l in (0, 47):
        x = synth.prompt(w.seed, l, w.prompt_T, w.H)
        y = st.forward(x, l)
        ids, _ = orc.route(x, st.router[l], st.bias)
        plan = orc.plan(l, ids, w.prompt_T)
        rec = st.cache.trace_read()[0]
        assert np.array_equal(rec["ids"], ids.reshape(-1))
        assert np.array_equal(rec["hit_of"].astype(np.uint8), plan["hit_of"])
        assert rec["n_hit"] == plan["n_hit"] and rec["n_uniq"] == plan["n_uniq"]
        # the layer output is per token: check a sample of tokens with the oracle
        tok = np.array([0, 1, 777, 1500, w.prompt_T - 1])
        _, _, yo = orc.layer(x[tok], st.router[l], st.bias, l)
        assert rel_l2(y[tok], yo) <= TOL
    after = st.cache.state()
    for key in before:
        assert np.array_equal(before[key], after[key])
    st.close()
