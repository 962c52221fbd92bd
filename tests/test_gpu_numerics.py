"""GPU numerics at the edges of the inputs, through the C ABI, against the oracle.

- The full-softmax weights (norm_topk = 0, the alternative reading of the
  combine weights) on the one-kernel decode, the three-kernel decode and the
  prefill path; each call must also differ clearly from the renormalised
  weights, so the test can tell the two readings apart.
- Hidden sizes that are multiples of 64 but not of 256 (the router reads
  256-column rounds per warp; the last round is partial).
- Token rows far outside fp16's range (1e-6 .. 1e6, a row mixing 1e4 and
  1e-4, a zero row): the expert kernels take fp16 operands after an exact
  power-of-two prescale of each token row and each activation row.

Routing, slots and hits are compared bit for bit on every call; outputs must
be within relative L2 1e-3 of the oracle's fp64 layer, per token where token
magnitudes differ.
"""
import numpy as np
import pytest

import oracle
import synth
from harness import OracleRun, Setup, compare_trace, cuda_available, rel_l2, rel_l2_rows, scale_bf16_rows
from synth.workloads import WORKLOADS, scaled

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

TOL = 1e-3


def decode_call(st, orc, x, layer, per_row=False):
    """One decode call: trace bit-exact against the oracle's routing and plan,
    output within TOL (per token if per_row). Returns (gpu, oracle) outputs."""
    T = x.shape[0]
    y = st.forward(x, layer)
    ids, _ = orc.route(x, st.router[layer], st.bias)
    compare_trace(st.cache.trace_read()[0], ids, orc.plan(layer, ids, T), layer, T)
    _, _, yo = orc.layer(x, st.router[layer], st.bias, layer)
    errs = rel_l2_rows(y, yo) if per_row else [rel_l2(y, yo)]
    assert max(errs) <= TOL, errs
    return y, yo


def prefill_call(st, orc, x, layer, per_row=False):
    """One prefill call (T above the cache limit): ids, hit flags and slots as
    the oracle's read-only lookup gives them, output within TOL."""
    T = x.shape[0]
    y = st.forward(x, layer)
    ids, _ = orc.route(x, st.router[layer], st.bias)
    plan = orc.plan(layer, ids, T)
    rec = st.cache.trace_read()[0]
    assert np.array_equal(rec["ids"], ids.reshape(-1))
    assert np.array_equal(rec["hit_of"].astype(np.uint8), plan["hit_of"])
    assert np.array_equal(rec["slot_of"], plan["slot_of"])
    _, _, yo = orc.layer(x, st.router[layer], st.bias, layer)
    errs = rel_l2_rows(y, yo) if per_row else [rel_l2(y, yo)]
    assert max(errs) <= TOL, errs
    return y, yo


# ---------------------------------------------------------------------------
# norm_topk = 0: weights are the softmax over all experts, read at the picks
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("decode,T", [("one_kernel", 1), ("one_kernel", 3), ("three_kernels", 1),
                                      ("three_kernels", 5)])
def test_full_softmax_weights_on_the_decode_paths(decode, T):
    w = scaled(WORKLOADS["flash_next_nvfp4"], name="norm0", L=2, E=64, k=4, H=512, I=192, fmt="q4_0",
               pool_mode="per_layer", slots_per_layer=24, pool_bytes=0.0, has_shared=True, bias=True,
               streams=(T,), steps=4, rho=0.7)
    st = Setup(w, decode=decode, norm_topk=False)
    orc = OracleRun(w, st.info["slot_bytes"], norm=False)
    ren = OracleRun(w, st.info["slot_bytes"])  # the renormalised reading
    xs = {l: st.hiddens(l, T, w.steps) for l in range(w.L)}
    for step in range(w.steps):
        for l in range(w.L):
            y, _ = decode_call(st, orc, xs[l][step], l)
            _, _, yr = ren.layer(xs[l][step], st.router[l], st.bias, l)
            assert rel_l2(y, yr) > 1e-2
    info = st.cache.info()
    calls = w.steps * w.L
    assert info["fused_decode_calls" if decode == "one_kernel" else "split_decode_calls"] == calls
    st.close()


def test_full_softmax_weights_on_the_prefill_path():
    T = 80
    w = scaled(WORKLOADS["flash_next_prefill"], name="norm0p", L=2, E=48, k=4, H=256, I=128, pool_mode="shared",
               pool_bytes=0.0, streams=(2,), steps=3, prompt_T=T)
    w = scaled(w, pool_bytes=oracle.slot_bytes(w.fmt, w.H, w.I) * 20)
    st = Setup(w, max_tokens=T, norm_topk=False)
    orc = OracleRun(w, st.info["slot_bytes"], norm=False)
    ren = OracleRun(w, st.info["slot_bytes"])
    for l in range(w.L):  # some decode calls first, so some experts are resident
        for x in st.hiddens(l, 2, w.steps):
            decode_call(st, orc, x, l)
    for l in range(w.L):
        x = synth.prompt(w.seed, l, T, w.H)
        y, _ = prefill_call(st, orc, x, l)
        _, _, yr = ren.layer(x, st.router[l], st.bias, l)
        assert rel_l2(y, yr) > 1e-2
    st.close()


# ---------------------------------------------------------------------------
# Hidden sizes that are not multiples of 256
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("H", [64, 320])
@pytest.mark.parametrize("decode", ["one_kernel", "three_kernels"])
def test_hidden_sizes_with_a_partial_router_round(H, decode):
    w = scaled(WORKLOADS["qwen3_30b_a3b_q4_0"], name="htail", L=2, E=32, k=4, H=H, I=128, slots_per_layer=12,
               bias=True, streams=(2,), steps=4, rho=0.7)
    st = Setup(w, decode=decode, max_tokens=40)
    orc = OracleRun(w, st.info["slot_bytes"])
    xs = {l: st.hiddens(l, 2, w.steps) for l in range(w.L)}
    for step in range(w.steps):
        for l in range(w.L):
            decode_call(st, orc, xs[l][step], l)
    for l in range(w.L):
        prefill_call(st, orc, synth.prompt(w.seed, l, 40, w.H), l)
    info = st.cache.info()
    assert info["fused_decode_calls" if decode == "one_kernel" else "split_decode_calls"] == w.steps * w.L
    st.close()


# ---------------------------------------------------------------------------
# Token rows outside fp16's range
# ---------------------------------------------------------------------------
def magnitude_rows(T, H, step):
    """Row factors of one call: huge, tiny, ordinary and zero rows, and (step 2)
    a row mixing 1e4 and 1e-4 column by column."""
    base = [[1e6, 1e-6, 1.0, 3e5], [2e-5, 7e4, 0.0, 1e6], [1.0, 1e-6, 5e5, 1.0]][step % 3][:T]
    f = np.repeat(np.asarray(base, dtype=np.float64)[:, None], H, axis=1)
    if step % 3 == 2:
        f[0, 0::2] = 1e4
        f[0, 1::2] = 1e-4
    return f


@pytest.mark.parametrize("fmt", ["q4_0", "fp8_b128", "nvfp4", "bf16"])
@pytest.mark.parametrize("decode", ["one_kernel", "three_kernels"])
def test_decode_token_rows_far_outside_fp16(fmt, decode):
    T = 4
    w = scaled(WORKLOADS["flash_next_nvfp4"], name="range", L=2, E=32, k=4, H=256, I=128, fmt=fmt,
               pool_mode="per_layer", slots_per_layer=16, pool_bytes=0.0, has_shared=fmt in ("q4_0", "nvfp4"),
               bias=True, streams=(T,), steps=3, rho=0.7)
    st = Setup(w, decode=decode)
    orc = OracleRun(w, st.info["slot_bytes"])
    xs = {l: st.hiddens(l, T, w.steps) for l in range(w.L)}
    for step in range(w.steps):
        for l in range(w.L):
            x = scale_bf16_rows(xs[l][step], magnitude_rows(T, w.H, step))
            y, yo = decode_call(st, orc, x, l, per_row=True)
            assert np.all(np.isfinite(y))
    info = st.cache.info()
    assert info["fused_decode_calls" if decode == "one_kernel" else "split_decode_calls"] == w.steps * w.L
    st.close()


@pytest.mark.parametrize("fmt", ["q4_0", "fp8_b128", "nvfp4", "bf16"])
def test_prefill_token_rows_far_outside_fp16(fmt):
    T = 48
    w = scaled(WORKLOADS["flash_next_prefill"], name="rangep", L=1, E=32, k=4, H=256, I=128, fmt=fmt,
               pool_mode="shared", pool_bytes=0.0, has_shared=fmt in ("q4_0", "nvfp4"), bias=True, streams=(1,),
               steps=1, prompt_T=T)
    w = scaled(w, pool_bytes=oracle.slot_bytes(fmt, w.H, w.I) * 12)
    st = Setup(w, max_tokens=T)
    orc = OracleRun(w, st.info["slot_bytes"])
    for x in st.hiddens(0, 1, 6):  # a few decode calls make some experts resident
        decode_call(st, orc, x, 0)
    cyc = np.array([1e6, 1e-6, 1.0, 5e4, 3e-3, 1.3e5, 0.0, 2e-5])
    f = np.repeat(cyc[np.arange(T) % cyc.size][:, None], w.H, axis=1)
    f[3, 0::2], f[3, 1::2] = 1e4, 1e-4
    x = scale_bf16_rows(synth.prompt(w.seed, 0, T, w.H), f)
    y, _ = prefill_call(st, orc, x, 0, per_row=True)
    assert np.all(np.isfinite(y))
    st.close()
