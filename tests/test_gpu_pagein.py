"""Page-in prefill ("Running an MoE Model Larger Than Your VRAM: SGLang Paged
Experts, ...", "Why do short prompts get slower first tokens?": a prefill
pages in everything it routes to that is not resident, once).

Every call's routing, slots, hits and fills, and the cache state after it,
must be those of the oracle's page-in mode (the decode transaction over all
of the prefill's distinct experts, without the capacity rule), including
prefills with more distinct experts than slots. Each occupied slot must hold
its expert's record, and every output must be bitwise that of a read-only
handle given the same calls (paging moves bytes, not results) and within
rel-L2 1e-3 of the oracle.
"""
import numpy as np
import pytest

import oracle
import synth
from harness import OracleRun, Setup, compare_trace, cuda_available, rel_l2
from synth.workloads import WORKLOADS, scaled

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

TOL = 1e-3


@pytest.mark.parametrize("fmt,pool_mode,K", [("nvfp4", "shared", 30), ("q4_0", "per_layer", 12),
                                             ("bf16", "per_layer", 20), ("fp8_b128", "shared", 64)])
def test_page_in_prefill_matches_the_oracle(fmt, pool_mode, K):
    T = 40
    w = scaled(WORKLOADS["flash_next_prefill"], name="pagein", L=2, E=48, k=4, H=256, I=128, fmt=fmt,
               pool_mode=pool_mode, slots_per_layer=K, pool_bytes=0.0, has_shared=fmt in ("nvfp4", "q4_0"),
               bias=True, streams=(2,), steps=3, prompt_T=T)
    if pool_mode == "shared":
        w = scaled(w, pool_bytes=oracle.slot_bytes(fmt, w.H, w.I) * K + 5)
    st = Setup(w, max_tokens=T, prefill="page_in")
    ro = Setup(w, max_tokens=T)
    orc = OracleRun(w, st.info["slot_bytes"], prefill="page_in")
    wrapped = False
    for r in range(3):
        calls = [(l, x) for l in range(w.L) for x in st.hiddens(l, 2, w.steps)]
        calls += [(l, synth.prompt(w.seed + 1000 * r, l, T, w.H)) for l in range(w.L)]
        for l, x in calls:
            y = st.forward(x, l)
            y_ro = ro.forward(x, l)
            assert np.array_equal(y, y_ro)
            rec = st.cache.trace_read()[0]
            ro.cache.trace_read()
            ids, _ = orc.route(x, st.router[l], st.bias)
            plan = orc.plan(l, ids, x.shape[0])
            compare_trace(rec, ids, plan, l, x.shape[0])
            wrapped |= plan["n_fill"] > orc.K
            if x.shape[0] > 32 or r == 0:
                _, _, yo = orc.layer(x, st.router[l], st.bias, l)
                assert rel_l2(y, yo) <= TOL
            if x.shape[0] > 32:
                g, o = st.cache.state(), orc.cache.state()
                for key in ("slot_map", "key_of", "order"):
                    assert np.array_equal(g[key], o[key]), key
                for p in range(g["key_of"].shape[0]):
                    for s, key in enumerate(g["key_of"][p]):
                        if key >= 0:
                            dev, store = st.cache.read_slot(p, s, key // w.E, key % w.E)
                            assert np.array_equal(dev, store), (p, s, key)
    if pool_mode == "per_layer" and K < w.E // 2:
        assert wrapped  # some prefill paged in more experts than its pool has slots
    gs, os_ = st.cache.stats(), orc.cache.stats()
    for b in range(3):
        for key, okey in (("calls", "calls"), ("hits", "hits"), ("misses", "misses"), ("bytes_uploaded", "bytes")):
            assert gs["buckets"][b][key] == os_[b][okey], (b, key)
    st.close()
    ro.close()
