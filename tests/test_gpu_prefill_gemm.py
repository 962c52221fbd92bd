"""GPU parity of the prefill expert FFN on the tensor cores (tcgen05 grouped
GEMMs, accumulators in tensor memory) against the oracle's unpaged fp64
layer, for the three quantised formats.

The shapes span several 128-row weight tiles (gate/up and down), several
128-pair token tiles per expert with ragged tails (a Zipf router bias gives
the popular experts hundreds of tokens), and both the resident experts read
in place and the staged ones copied through the arena.
"""
import numpy as np
import pytest

import synth
from harness import OracleRun, Setup, compare_trace, cuda_available, rel_l2
from synth.workloads import WORKLOADS, scaled

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

TOL = 1e-3


@pytest.mark.parametrize("fmt", ["nvfp4", "q4_0", "fp8_b128"])
def test_prefill_grouped_gemm_matches_oracle(fmt):
    T = 300
    w = scaled(WORKLOADS["flash_next_prefill"], name="gemm", L=1, E=16, k=4, H=512, I=256, fmt=fmt,
               pool_mode="per_layer", slots_per_layer=8, pool_bytes=0.0, has_shared=True, bias=True,
               streams=(1,), steps=4, prompt_T=T)
    st = Setup(w, max_tokens=T)
    orc = OracleRun(w, st.info["slot_bytes"])
    # a few decode calls leave some experts resident (read in place by the
    # prefill); the rest are staged through the arena
    xs = st.hiddens(0, 1, w.steps)
    for s in range(w.steps):
        st.forward(xs[s], 0)
        ids, _ = orc.route(xs[s], st.router[0], st.bias)
        orc.plan(0, ids, 1)
        st.cache.trace_read()
    x = synth.prompt(w.seed, 0, T, w.H)
    y = st.forward(x, 0)
    ids, _ = orc.route(x, st.router[0], st.bias)
    plan = orc.plan(0, ids, T)
    rec = st.cache.trace_read()[0]
    assert np.array_equal(rec["ids"], ids.reshape(-1))
    assert np.array_equal(rec["hit_of"].astype(np.uint8), plan["hit_of"])
    assert 0 < rec["n_hit"] < rec["n_uniq"]  # both read-in-place and staged experts
    counts = np.bincount(ids.reshape(-1), minlength=w.E)
    assert counts.max() > 128 and (counts % 128 != 0).any()  # several tiles per expert, ragged tails
    _, _, yo = orc.layer(x, st.router[0], st.bias, 0)
    err = rel_l2(y, yo)
    assert err <= TOL, err
    # every token, not only the whole prompt
    per_tok = np.linalg.norm(y - yo, axis=1) / np.linalg.norm(yo, axis=1)
    assert per_tok.max() <= 4 * TOL, per_tok.max()
    st.close()


def test_prefill_leaves_decode_state_and_results_unchanged():
    # A prefill between decode steps neither changes the LRU state nor the
    # decode outputs that follow (the GEMM path writes only its own scratch).
    T = 200
    w = scaled(WORKLOADS["flash_next_prefill"], name="gemm2", L=2, E=16, k=4, H=256, I=128, fmt="nvfp4",
               pool_mode="shared", pool_bytes=0.0, has_shared=True, bias=True, streams=(2,), steps=6,
               prompt_T=T)
    import oracle
    w = scaled(w, pool_bytes=oracle.slot_bytes(w.fmt, w.H, w.I) * 12)
    outs = []
    for with_prefill in (False, True):
        st = Setup(w, max_tokens=T)
        orc = OracleRun(w, st.info["slot_bytes"])
        xs = {l: st.hiddens(l, 2, w.steps) for l in range(w.L)}
        ys = []
        for s in range(w.steps):
            if with_prefill and s == 3:
                before = st.cache.state()
                for l in range(w.L):
                    st.forward(synth.prompt(w.seed, l, T, w.H), l)
                    st.cache.trace_read()
                after = st.cache.state()
                for key in before:
                    assert np.array_equal(before[key], after[key])
            for l in range(w.L):
                ys.append(st.forward(xs[l][s], l))
                ids, _ = orc.route(xs[l][s], st.router[l], st.bias)
                plan = orc.plan(l, ids, 2)
                compare_trace(st.cache.trace_read()[0], ids, plan, l, 2)
        outs.append(np.stack(ys))
        st.close()
    assert np.array_equal(outs[0], outs[1])
