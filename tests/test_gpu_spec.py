"""Speculative next-layer routing and prefetch ("Running a 133 GB MoE model on
an 8 GB GPU at 11 tokens/s by streaming experts from NVMe", "Workflow": run the
next layer's router on the current layer's input and start the predicted
experts' copies one layer early).

Speculation may only move bytes: with it on, every call's routing, slots,
hits and fills, every output, the final cache state and the counters must be
bitwise those of the same calls with it off, and match the oracle. The
inputs chain the layers (layer l + 1's tokens are layer l's, perturbed), so
the predictions are mostly right and the bank is read.
"""
import numpy as np
import pytest

from harness import OracleRun, Setup, compare_trace, cuda_available, rel_l2
from synth.workloads import WORKLOADS, scaled

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

TOL = 1e-3


def chained_inputs(st, T, steps, keep):
    """[steps][L] token rows: layer 0 draws its AR(1) stream; layer l + 1 keeps
    the fraction `keep` of layer l's columns and takes the rest from its own
    stream, so the next layer's router sees nearly its own input."""
    w = st.w
    own = {l: st.hiddens(l, T, steps) for l in range(w.L)}
    rng = np.random.default_rng(7)
    out = []
    for s in range(steps):
        row = [own[0][s]]
        for l in range(1, w.L):
            x = own[l][s].copy()
            m = rng.random(w.H) < keep
            x[:, m] = row[-1][:, m]
            row.append(x)
        out.append(row)
    return out


def run(w, spec, xs, order, T, decode="auto"):
    st = Setup(w, speculate=spec, decode=decode)
    orc = OracleRun(w, st.info["slot_bytes"])
    ys, recs = [], []
    for s, row in enumerate(xs):
        for l in order:
            y = st.forward(row[l], l)
            rec = st.cache.trace_read()[0]
            ids, _ = orc.route(row[l], st.router[l], st.bias)
            compare_trace(rec, ids, orc.plan(l, ids, T), l, T)
            if s % 3 == 0:
                _, _, yo = orc.layer(row[l], st.router[l], st.bias, l)
                assert rel_l2(y, yo) <= TOL
            ys.append(y)
            recs.append(rec)
    res = (np.stack(ys), recs, st.cache.state(), st.cache.stats(), st.cache.info())
    st.close()
    return res


@pytest.mark.parametrize("fmt,pool_mode,T", [("nvfp4", "shared", 1), ("q4_0", "per_layer", 2),
                                             ("fp8_b128", "per_layer", 1)])
def test_speculation_moves_bytes_only(fmt, pool_mode, T):
    import oracle
    w = scaled(WORKLOADS["flash_next_nvfp4"], name="spec", L=4, E=64, k=4, H=512, I=192, fmt=fmt,
               pool_mode=pool_mode, slots_per_layer=10, pool_bytes=0.0, has_shared=fmt != "fp8_b128", bias=True,
               streams=(T,), steps=8, rho=0.6)
    if pool_mode == "shared":
        w = scaled(w, pool_bytes=oracle.slot_bytes(fmt, w.H, w.I) * 24 + 5)
    probe = Setup(w)
    xs = chained_inputs(probe, T, w.steps, keep=0.9)
    probe.close()
    order = list(range(w.L))
    y0, r0, s0, c0, i0 = run(w, False, xs, order, T)
    y1, r1, s1, c1, i1 = run(w, True, xs, order, T)
    assert np.array_equal(y0, y1)
    for a, b in zip(r0, r1):
        for key in ("ids", "slot_of", "hit_of", "fill_expert", "fill_slot"):
            assert np.array_equal(a[key], b[key]), key
    for key in s0:
        assert np.array_equal(s0[key], s1[key]), key
    for b in range(3):
        for key in ("calls", "hits", "misses", "bytes_uploaded"):
            assert c0["buckets"][b][key] == c1["buckets"][b][key]
    assert c0["spec_prefetched"] == 0 and c0["spec_used"] == 0
    assert c1["spec_prefetched"] > 0 and 0 < c1["spec_used"] <= c1["spec_prefetched"]
    assert i1["fused_decode_calls"] == 0  # speculation takes the three-kernel path


def test_speculation_with_layers_out_of_order_and_an_unregistered_router():
    # calls that skip or repeat layers join the side stream's work first; a
    # layer without a registered router is never predicted
    import torch
    w = scaled(WORKLOADS["qwen3_30b_a3b_q4_0"], name="spec_order", L=4, E=32, k=4, H=256, I=128,
               slots_per_layer=8, bias=True, streams=(1,), steps=6, rho=0.5)
    probe = Setup(w)
    xs = chained_inputs(probe, 1, w.steps, keep=1.0)
    probe.close()
    order = [0, 1, 3, 2, 0, 1, 2, 3, 2, 3]
    y0, r0, s0, c0, _ = run(w, False, xs, order, 1)
    st = Setup(w, speculate=True)
    st.cache.set_router(2, None)  # layer 2 is never predicted
    orc = OracleRun(w, st.info["slot_bytes"])
    ys = []
    for row in xs:
        for l in order:
            ys.append(st.forward(row[l], l))
            ids, _ = orc.route(row[l], st.router[l], st.bias)
            compare_trace(st.cache.trace_read()[0], ids, orc.plan(l, ids, 1), l, 1)
    assert np.array_equal(np.stack(ys), y0)
    st1 = st.cache.stats()
    assert st1["spec_prefetched"] > 0
    st.close()
