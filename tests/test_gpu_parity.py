"""GPU parity: the CUDA path through the C ABI against the oracle.

Routing (top-k ids in rank order), slot assignments, hit flags and fills are
compared bit for bit on every call; layer outputs (fp32) must be within
relative L2 1e-3 of the oracle's fp64 unpaged layer on every call.
"""
import numpy as np
import pytest

from harness import OracleRun, Setup, compare_trace, cuda_available, rel_l2
from synth.workloads import WORKLOADS, scaled

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

TOL = 1e-3


def run_steps(st, orc, steps, T, layers=None, check_out=True, out_every=1):
    w = st.w
    layers = range(w.L) if layers is None else layers
    xs = {l: st.hiddens(l, T, steps) for l in layers}
    worst = 0.0
    for step in range(steps):
        for l in layers:
            x = xs[l][step]
            y = st.forward(x, l)
            ids, _ = orc.route(x, st.router[l], st.bias)
            plan = orc.plan(l, ids, T)
            recs = st.cache.trace_read()
            assert len(recs) == 1
            compare_trace(recs[0], ids, plan, l, T)
            if check_out and step % out_every == 0:
                _, _, yo = orc.layer(x, st.router[l], st.bias, l)
                err = rel_l2(y, yo)
                worst = max(worst, err)
                assert err <= TOL, (step, l, err)
    return worst


def test_tiny_workload_full():
    w = WORKLOADS["tiny"]
    st = Setup(w)
    orc = OracleRun(w, st.info["slot_bytes"])
    worst = run_steps(st, orc, w.steps, w.streams[0])
    g = st.cache.state()
    o = orc.cache.state()
    assert np.array_equal(g["slot_map"], o["slot_map"])
    assert np.array_equal(g["key_of"], o["key_of"])
    assert np.array_equal(g["order"], o["order"])
    gs, os_ = st.cache.stats(), orc.cache.stats()
    for b in range(3):
        for key, okey in (("calls", "calls"), ("hits", "hits"), ("misses", "misses"), ("bytes_uploaded", "bytes")):
            assert gs["buckets"][b][key] == os_[b][okey], (b, key)
    print("tiny worst rel-L2", worst)
    st.close()


@pytest.mark.parametrize("fmt", ["bf16", "q4_0", "fp8_b128", "nvfp4"])
@pytest.mark.parametrize("pool_mode", ["per_layer", "shared"])
def test_formats_small(fmt, pool_mode):
    base = WORKLOADS["flash_next_nvfp4"]
    # 3 layers, 40 experts top-4, H 512, I 192 (3 row chunks of 64 + ragged
    # tile counts), tight pools so evictions happen every step
    w = scaled(base, name="small", L=3, E=40, k=4, H=512, I=192, fmt=fmt, pool_mode=pool_mode,
               slots_per_layer=14, pool_bytes=0.0, has_shared=(fmt in ("nvfp4", "q4_0")), bias=True,
               streams=(3,), steps=10, rho=0.7)
    from harness import pool_slots  # noqa
    import oracle
    sb = oracle.slot_bytes(fmt, w.H, w.I)
    if pool_mode == "shared":
        w = scaled(w, pool_bytes=sb * 16 + 5)
    st = Setup(w)
    assert st.info["slot_bytes"] == sb
    orc = OracleRun(w, st.info["slot_bytes"])
    worst = run_steps(st, orc, w.steps, 3)
    g, o = st.cache.state(), orc.cache.state()
    assert np.array_equal(g["order"], o["order"]) and np.array_equal(g["slot_map"], o["slot_map"])
    print(fmt, pool_mode, "worst rel-L2", worst)
    st.close()


@pytest.mark.parametrize("T", [1, 2, 5, 8, 17, 32])
def test_token_counts(T):
    w = scaled(WORKLOADS["qwen3_30b_a3b_q4_0"], name="tok", L=2, E=64, k=8, H=256, I=128,
               slots_per_layer=max(8 * T, 20), steps=3, streams=(T,))
    st = Setup(w, max_tokens=32)
    orc = OracleRun(w, st.info["slot_bytes"])
    run_steps(st, orc, 3, T)
    st.close()


def test_paging_invariance_across_pool_sizes():
    # The same calls with every expert resident, with the configured pool and
    # with the smallest legal pool give bitwise identical outputs.
    w = scaled(WORKLOADS["qwen3_30b_a3b_fp8"], name="inv", L=2, E=24, k=4, H=256, I=128, streams=(2,), steps=8)
    outs = []
    for K in (24, 12, 8):
        st = Setup(w, K=K, trace=0)
        xs = {l: st.hiddens(l, 2, w.steps) for l in range(w.L)}
        ys = [st.forward(xs[l][s], l) for s in range(w.steps) for l in range(w.L)]
        outs.append(np.stack(ys))
        st.close()
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_upload_modes_agree_and_slots_hold_the_store_bytes():
    w = scaled(WORKLOADS["qwen3_30b_a3b_q4_0"], name="upl", L=2, E=24, k=4, H=256, I=128, streams=(2,), steps=6,
               slots_per_layer=9)
    res = {}
    for mode in ("pull", "memcpy"):
        st = Setup(w, upload=mode)
        orc = OracleRun(w, st.info["slot_bytes"])
        xs = {l: st.hiddens(l, 2, w.steps) for l in range(w.L)}
        ys = []
        for s in range(w.steps):
            for l in range(w.L):
                ys.append(st.forward(xs[l][s], l))
                ids, _ = orc.route(xs[l][s], st.router[l], st.bias)
                plan = orc.plan(l, ids, 2)
                rec = st.cache.trace_read()[0]
                compare_trace(rec, ids, plan, l, 2)
        res[mode] = np.stack(ys)
        # every occupied slot holds its expert's store bytes exactly
        state = st.cache.state()
        for p in range(state["key_of"].shape[0]):
            for s, key in enumerate(state["key_of"][p]):
                if key < 0:
                    continue
                dev_bytes, store_bytes = st.cache.read_slot(p, s, key // w.E, key % w.E)
                assert np.array_equal(dev_bytes, store_bytes), (mode, p, s, key)
        stats = st.cache.stats()
        assert stats["buckets"][0]["misses"] > 0 and stats["buckets"][0]["upload_ns"] > 0
        st.close()
    assert np.array_equal(res["pull"], res["memcpy"])


def test_prefill_path_reads_in_place_and_keeps_the_lru():
    w = scaled(WORKLOADS["flash_next_prefill"], name="pre", L=2, E=48, k=4, H=256, I=128, pool_mode="shared",
               pool_bytes=0.0, streams=(2,), steps=4, prompt_T=80)
    import oracle
    import synth
    sb = oracle.slot_bytes(w.fmt, w.H, w.I)
    w = scaled(w, pool_bytes=sb * 20)
    st = Setup(w, max_tokens=80)
    orc = OracleRun(w, st.info["slot_bytes"])
    # warm the cache with a few decode calls
    run_steps(st, orc, 3, 2, check_out=False)
    before = st.cache.state()
    for l in range(w.L):
        x = synth.prompt(w.seed, l, 80, w.H)
        y = st.forward(x, l)
        ids, _ = orc.route(x, st.router[l], st.bias)
        plan = orc.plan(l, ids, 80)
        rec = st.cache.trace_read()[0]
        assert np.array_equal(rec["ids"], ids.reshape(-1))
        assert np.array_equal(rec["hit_of"].astype(np.uint8), plan["hit_of"])
        assert np.array_equal(rec["slot_of"], plan["slot_of"])
        _, _, yo = orc.layer(x, st.router[l], st.bias, l)
        assert rel_l2(y, yo) <= TOL
    after = st.cache.state()
    for key in before:
        assert np.array_equal(before[key], after[key])
    s = st.cache.stats()["buckets"][2]
    o = orc.cache.stats()[2]
    assert s["calls"] == o["calls"] == 2 and s["hits"] == o["hits"] and s["misses"] == o["misses"]
    st.close()


def test_capacity_rule_refuses_without_changing_state():
    import paged_expert_cache_gb300 as pec
    w = scaled(WORKLOADS["tiny"], name="cap", steps=2, streams=(4,))
    st = Setup(w, max_tokens=8)
    x = st.hiddens(0, 4, 1)[0]
    st.forward(x, 0)
    before = st.cache.state()
    x5 = st.hiddens(0, 5, 1)[0]  # 5 tokens * top-2 = 10 > 8 slots
    with pytest.raises(pec.MoeError) as ei:
        st.forward(x5, 0)
    assert ei.value.status == pec.ERR_CAPACITY
    after = st.cache.state()
    for key in before:
        assert np.array_equal(before[key], after[key])
    st.close()


def test_exact_ties_rank_the_lower_expert_first():
    import torch
    w = scaled(WORKLOADS["tiny"], name="ties", E=16, k=4, steps=4, streams=(3,), bias=False, slots_per_layer=12)
    st = Setup(w)
    # duplicate router rows: experts (3, 9) and (5, 12) tie on every input
    r = st.router[0].copy()
    r[9] = r[3]
    r[12] = r[5]
    st.router[0] = r
    st.router_dev[0] = torch.from_numpy(r.view(np.int16)).to(st.dev)
    orc = OracleRun(w, st.info["slot_bytes"])
    run_steps(st, orc, 4, 3)
    assert st.cache.stats()["topk_fp64_rerank"] > 0
    st.close()


@pytest.mark.parametrize("pool_mode", ["per_layer", "shared"])
def test_multi_wave_decode_matches_the_oracle_wave_by_wave(pool_mode):
    # T * k above the pool's slots with multi_wave: waves of K // k tokens in
    # token order, each its own cache transaction and trace record, checked
    # against the oracle's wave split and literal LRU; the outputs match the
    # unpaged layer and, bit for bit, a pool large enough for one wave.
    import oracle
    T, K = 7, 10
    w = scaled(WORKLOADS["tiny"], name="waves", L=2, E=16, k=4, steps=5, streams=(T,), bias=True,
               pool_mode=pool_mode, slots_per_layer=K, pool_bytes=0.0)
    sb = oracle.slot_bytes(w.fmt, w.H, w.I)
    if pool_mode == "shared":
        w = scaled(w, pool_bytes=sb * K + 5)
    waves = oracle.wave_split(T, w.k, K)
    assert len(waves) == 4
    outs = []
    for big in (False, True):
        st = Setup(w, multi_wave=True, max_tokens=T, K=(4 * K if big else None),
                   pool_bytes=(sb * 4 * K if big and pool_mode == "shared" else None))
        orc = OracleRun(w, st.info["slot_bytes"])
        xs = {l: st.hiddens(l, T, w.steps) for l in range(w.L)}
        ys = []
        for step in range(w.steps):
            for l in range(w.L):
                x = xs[l][step]
                y = st.forward(x, l)
                ys.append(y)
                recs = st.cache.trace_read()
                if big:
                    assert len(recs) == 1
                    continue
                assert len(recs) == len(waves)
                for rec, (s0, n) in zip(recs, waves):
                    ids, _ = orc.route(x[s0:s0 + n], st.router[l], st.bias)
                    compare_trace(rec, ids, orc.plan(l, ids, n), l, n)
                _, _, yo = orc.layer(x, st.router[l], st.bias, l)
                assert rel_l2(y, yo) <= TOL
        outs.append(np.stack(ys))
        st.close()
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("pool_mode", ["per_layer", "shared"])
def test_lfu_eviction_matches_the_oracle_on_both_decode_paths(pool_mode):
    # eviction LFU: every call's routing, slots, hits and fills bit-exact
    # against the oracle's LFU, on the one-kernel and the three-kernel paths
    # (which agree bit for bit), with a pool small enough to evict often; the
    # policy must also part from LRU somewhere on the way.
    import oracle
    w = scaled(WORKLOADS["tiny"], name="lfu", L=2, E=16, k=2, steps=24, streams=(2,), bias=True,
               pool_mode=pool_mode, slots_per_layer=5, pool_bytes=0.0, rho=0.5)
    if pool_mode == "shared":
        w = scaled(w, pool_bytes=oracle.slot_bytes(w.fmt, w.H, w.I) * 7 + 5)
    runs = {}
    for decode in ("one_kernel", "three_kernels"):
        st = Setup(w, decode=decode, eviction="lfu")
        orc = OracleRun(w, st.info["slot_bytes"], policy="lfu")
        lru = OracleRun(w, st.info["slot_bytes"])
        ys, parted = [], False
        for T in (1, 2):
            xs = {l: st.hiddens(l, T, w.steps) for l in range(w.L)}
            for step in range(w.steps):
                for l in range(w.L):
                    x = xs[l][step]
                    ys.append(st.forward(x, l))
                    ids, _ = orc.route(x, st.router[l], st.bias)
                    plan = orc.plan(l, ids, T)
                    compare_trace(st.cache.trace_read()[0], ids, plan, l, T)
                    parted |= not np.array_equal(lru.plan(l, ids, T)["slot_of"], plan["slot_of"])
                    if step % 6 == 0:
                        _, _, yo = orc.layer(x, st.router[l], st.bias, l)
                        assert rel_l2(ys[-1], yo) <= TOL
        assert parted
        runs[decode] = np.concatenate([y.reshape(-1) for y in ys])
        st.close()
    assert np.array_equal(runs["one_kernel"], runs["three_kernels"])


def test_exact_ties_one_token_on_both_decode_paths():
    # One token per call: the one-kernel path ranks with one thread per
    # expert and certifies with a block-wide AND; exact ties fail the
    # certificate and take the fp64 re-rank. Both paths must pick the lower
    # expert, match the oracle, and give the same bits.
    import torch
    w = scaled(WORKLOADS["tiny"], name="ties1", E=16, k=4, steps=16, streams=(1,), bias=False, slots_per_layer=12)
    outs = {}
    for mode in ("one_kernel", "three_kernels"):
        st = Setup(w, decode=mode)
        r = st.router[0].copy()
        r[9] = r[3]
        r[12] = r[5]
        r[14] = r[0]
        st.router[0] = r
        st.router_dev[0] = torch.from_numpy(r.view(np.int16)).to(st.dev)
        orc = OracleRun(w, st.info["slot_bytes"])
        xs = st.hiddens(0, 1, w.steps)
        ys = []
        for step in range(w.steps):
            ys.append(st.forward(xs[step], 0))
            ids, _ = orc.route(xs[step], st.router[0], st.bias)
            plan = orc.plan(0, ids, 1)
            compare_trace(st.cache.trace_read()[0], ids, plan, 0, 1)
            _, _, yo = orc.layer(xs[step], st.router[0], st.bias, 0)
            assert rel_l2(ys[-1], yo) <= TOL
        info = st.cache.info()
        assert info["fused_decode_calls" if mode == "one_kernel" else "split_decode_calls"] == w.steps
        assert st.cache.stats()["topk_fp64_rerank"] > 0
        outs[mode] = np.stack(ys)
        st.close()
    assert np.array_equal(outs["one_kernel"], outs["three_kernels"])


@pytest.mark.parametrize("fmt,pool_mode,E,T", [
    ("q4_0", "per_layer", 64, 1), ("q4_0", "shared", 64, 3), ("fp8_b128", "per_layer", 40, 8),
    ("nvfp4", "shared", 160, 2), ("bf16", "per_layer", 16, 4), ("nvfp4", "per_layer", 160, 4),
    ("nvfp4", "shared", 512, 1), ("q4_0", "per_layer", 300, 1)])
def test_one_kernel_and_three_kernel_decode_agree_bitwise(fmt, pool_mode, E, T):
    # The persistent one-kernel decode and the route / gate/up
    # / down kernels give the same bits: ids, slots, fills, outputs, final
    # state and counters; both match the oracle.
    k = 4 if E >= 40 else 2
    one_vs_three_kernels(fmt, pool_mode, E, T, k, H=512, I=192, L=3, steps=6, has_shared=fmt in ("nvfp4", "q4_0"))


@pytest.mark.parametrize("E,k", [(288, 12), (512, 16), (384, 16)])
def test_one_token_wide_ranking_threshold_and_merge(E, k):
    # One token over more than 256 experts: the persistent kernel ranks by a
    # threshold selection, or by the sorted-list merge when the candidates
    # overflow (288 experts fill 9 warps, fewer than k = 12 warp maxima, so
    # every key is a candidate); both agree with the three-kernel path and the
    # oracle.
    one_vs_three_kernels("nvfp4", "shared", E, 1, k, H=512, I=192, L=2, steps=5, has_shared=True)


@pytest.mark.parametrize("fmt,H,I,T,k,has_shared", [
    ("fp8_b128", 2048, 512, 8, 4, False),   # one ring slot
    ("q4_0", 2048, 512, 4, 8, False),       # three ring slots, refilled
    ("nvfp4", 2048, 768, 4, 4, True),       # three ring slots, shared expert
    ("bf16", 1024, 256, 2, 4, False)])      # three ring slots
def test_one_kernel_decode_with_a_small_ring(fmt, H, I, T, k, has_shared):
    # Large tiles leave room for one or three weight slots in shared memory,
    # so the two consumer groups of the one-kernel decode refill slots the
    # other group reads next; results stay those of the three kernels.
    one_vs_three_kernels(fmt, "per_layer", 64, T, k, H=H, I=I, L=2, steps=4, has_shared=has_shared)


def one_vs_three_kernels(fmt, pool_mode, E, T, k, H, I, L, steps, has_shared):
    w = scaled(WORKLOADS["flash_next_nvfp4"], name="fused", L=L, E=E, k=k, H=H, I=I, fmt=fmt,
               pool_mode=pool_mode, slots_per_layer=max(T * k + 3, 12), pool_bytes=0.0,
               has_shared=has_shared, bias=True, streams=(T,), steps=steps, rho=0.7)
    import oracle
    sb = oracle.slot_bytes(fmt, w.H, w.I)
    if pool_mode == "shared":
        w = scaled(w, pool_bytes=sb * (T * k + 6) + 5)
    runs = {}
    for split in (False, True):
        st = Setup(w, decode="three_kernels" if split else "one_kernel")
        orc = OracleRun(w, st.info["slot_bytes"])
        xs = {l: st.hiddens(l, T, w.steps) for l in range(w.L)}
        ys, recs = [], []
        for s in range(w.steps):
            for l in range(w.L):
                y = st.forward(xs[l][s], l)
                ids, _ = orc.route(xs[l][s], st.router[l], st.bias)
                plan = orc.plan(l, ids, T)
                rec = st.cache.trace_read()[0]
                compare_trace(rec, ids, plan, l, T)
                ys.append(y)
                recs.append(rec)
                if s % 3 == 0:
                    _, _, yo = orc.layer(xs[l][s], st.router[l], st.bias, l)
                    assert rel_l2(y, yo) <= TOL
        info = st.cache.info()
        calls = w.steps * w.L
        assert (info["split_decode_calls"], info["fused_decode_calls"]) == ((calls, 0) if split else (0, calls))
        runs[split] = (np.stack(ys), recs, st.cache.state(), st.cache.stats())
        st.close()
    (y0, r0, s0, c0), (y1, r1, s1, c1) = runs[False], runs[True]
    assert np.array_equal(y0, y1)
    for a, b in zip(r0, r1):
        for key in ("ids", "slot_of", "hit_of", "fill_expert", "fill_slot"):
            assert np.array_equal(a[key], b[key]), key
    for key in s0:
        assert np.array_equal(s0[key], s1[key]), key
    for bkt in range(3):
        for key in ("calls", "hits", "misses", "bytes_uploaded"):
            assert c0["buckets"][bkt][key] == c1["buckets"][bkt][key]
    if c0["buckets"][0]["misses"]:
        assert c0["buckets"][0]["upload_ns"] > 0


def test_decode_modes_choose_their_path_and_agree():
    # AUTO takes one kernel for one or two tokens on per-layer pools and three
    # kernels for three; ONE_KERNEL and THREE_KERNELS force the path. Every
    # mode gives the same bits.
    w = scaled(WORKLOADS["qwen3_30b_a3b_q4_0"], name="modes", L=2, E=32, k=4, H=512, I=192, slots_per_layer=16,
               streams=(3,), steps=3, rho=0.7)
    outs = {}
    for mode in ("auto", "one_kernel", "three_kernels"):
        st = Setup(w, decode=mode)
        ys = []
        for T in (1, 2, 3):
            xs = {l: st.hiddens(l, T, w.steps) for l in range(w.L)}
            for s in range(w.steps):
                for l in range(w.L):
                    ys.append(st.forward(xs[l][s], l).copy())
        info = st.cache.info()
        outs[mode] = (np.concatenate([y.reshape(-1) for y in ys]), info["fused_decode_calls"], info["split_decode_calls"])
        st.close()
    per_T = w.steps * w.L
    assert outs["auto"][1:] == (2 * per_T, per_T)
    assert outs["one_kernel"][1:] == (3 * per_T, 0)
    assert outs["three_kernels"][1:] == (0, 3 * per_T)
    assert np.array_equal(outs["auto"][0], outs["one_kernel"][0])
    assert np.array_equal(outs["auto"][0], outs["three_kernels"][0])
