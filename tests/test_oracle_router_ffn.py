"""Pins for the oracle's router, top-k, weights and expert FFN (CPU only)."""
import math
from fractions import Fraction

import numpy as np
import torch

import oracle
import synth


def _bf16(vals):
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bf16_values(bits):
    return torch.from_numpy(np.asarray(bits).view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def test_logits_one_hot_is_a_router_column_plus_bias():
    E, H = 12, 64
    W = synth.router_weights(3, 0, E, H)
    b = synth.zipf_bias(E)
    for h in (0, 17, 63):
        x = _bf16([1.0 if j == h else 0.0 for j in range(H)])[None, :]
        z = oracle.router_logits(x, W, b)[0]
        want = _bf16_values(W[:, h]) + b.astype(np.float64)
        assert np.array_equal(z, want)


def test_logits_exact_on_small_ints_and_close_to_rational_sum():
    rng = np.random.default_rng(1)
    E, H, T = 5, 40, 3
    xv = rng.integers(-8, 9, size=(T, H)).astype(np.float32)
    wv = rng.integers(-8, 9, size=(E, H)).astype(np.float32)
    z = oracle.router_logits(_bf16(xv), _bf16(wv))
    assert np.array_equal(z, xv.astype(np.float64) @ wv.astype(np.float64).T)
    # random bf16 values: the fp64 sum differs from the exact rational sum by
    # at most gamma_{H-1} * sum|x w| (sequential summation bound)
    W = synth.router_weights(9, 0, E, 2048)
    X = synth.hidden_ar1(9, 0, 0, T, 2048, 0.9)
    z = oracle.router_logits(X, W)
    xd, wd = _bf16_values(X), _bf16_values(W)
    u = 2.0 ** -53
    for t in range(T):
        for e in range(E):
            exact = sum(Fraction(float(a)) * Fraction(float(c)) for a, c in zip(xd[t], wd[e]))
            absum = float(np.sum(np.abs(xd[t] * wd[e])))
            bound = (2047 * u / (1 - 2047 * u)) * absum
            assert abs(Fraction(z[t, e]) - exact) <= Fraction(bound)


def test_topk_ties_go_to_the_lower_index():
    H = 32
    base = synth.router_weights(4, 0, 6, H)
    W = base.copy()
    W[4] = W[1]  # experts 1 and 4 tie on every input
    W[5] = W[2]
    x = synth.hidden_ar1(4, 0, 0, 5, H, 0.5)
    z = oracle.router_logits(x, W)
    ids, _ = oracle.topk(z, 6)
    for t in range(5):
        r = list(ids[t])
        assert r.index(1) < r.index(4) and r.index(2) < r.index(5)
        assert r.index(4) == r.index(1) + 1 and r.index(5) == r.index(2) + 1
    # all-equal logits: ranks are 0..k-1 and weights 1/k
    z = np.zeros((1, 9))
    ids, w = oracle.topk(z, 4)
    assert list(ids[0]) == [0, 1, 2, 3] and np.allclose(w, 0.25, rtol=0, atol=1e-15)


def test_topk_matches_a_lexicographic_sort():
    rng = np.random.default_rng(2)
    z = np.round(rng.normal(size=(50, 40)), 1)  # many exact ties
    ids, _ = oracle.topk(z, 7)
    for t in range(50):
        order = np.lexsort((np.arange(40), -z[t]))[:7]
        assert np.array_equal(ids[t], order)


def test_weights_renormalised_and_full_softmax():
    rng = np.random.default_rng(3)
    z = rng.normal(size=(4, 20))
    ids, w = oracle.topk(z, 5, norm=True)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-15)
    for t in range(4):
        sel = z[t, ids[t]]
        ref = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
        assert np.allclose(w[t], ref, rtol=1e-15, atol=0)
    ids1, w1 = oracle.topk(z, 1, norm=True)
    assert np.all(w1 == 1.0)
    ids0, w0 = oracle.topk(z, 5, norm=False)
    p = np.exp(z - z.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    assert np.array_equal(ids0, ids)
    assert np.allclose(w0, np.take_along_axis(p, ids, 1), rtol=1e-14, atol=0)


def _silu(v):
    return v / (1.0 + math.exp(-v))


def test_ffn_identity_weights_closed_form():
    # H = I, gate = up = down = identity (bf16): y = silu(x) * x elementwise
    H = I = 32
    eye = _bf16(np.eye(H, dtype=np.float32)).reshape(-1)
    rec = np.concatenate([eye.view(np.uint8)] * 3)
    x = np.linspace(-3, 3, H)
    y = oracle.expert_ffn("bf16", rec, H, I, x)
    want = np.array([_silu(v) * v for v in x])
    assert np.allclose(y, want, rtol=1e-15, atol=0)
    assert np.all(oracle.expert_ffn("bf16", rec, H, I, np.zeros(H)) == 0.0)


def test_ffn_gate_and_up_are_not_swapped():
    # gate = 2*I, up = 3*I, down = I: y = silu(2x) * 3x, which is not
    # silu(3x) * 2x, so a swap of the two matrices fails here
    H = I = 16
    eye = np.eye(H, dtype=np.float32)
    rec = np.concatenate([_bf16(2 * eye).reshape(-1).view(np.uint8), _bf16(3 * eye).reshape(-1).view(np.uint8),
                          _bf16(eye).reshape(-1).view(np.uint8)])
    x = np.linspace(-2, 2, H)
    y = oracle.expert_ffn("bf16", rec, H, I, x)
    want = np.array([_silu(2 * v) * 3 * v for v in x])
    assert np.allclose(y, want, rtol=1e-15, atol=0)


def test_ffn_rectangular_matches_library_matmul():
    # non-square shapes catch a transposed down projection
    for fmt in ("bf16", "q4_0", "fp8_b128", "nvfp4"):
        H, I = 256, 128
        rec = synth.expert_record(fmt, 11, 2, 5, H, I)
        mgu, mdn = oracle.matrix_bytes(fmt, I, H), oracle.matrix_bytes(fmt, H, I)
        g = np.frombuffer(rec[2 * mgu + mdn:].tobytes(), dtype=np.float32) if fmt == "nvfp4" else [1.0] * 3
        Wg = oracle.dequant_matrix(fmt, rec[:mgu], I, H, g[0])
        Wu = oracle.dequant_matrix(fmt, rec[mgu:2 * mgu], I, H, g[1])
        Wd = oracle.dequant_matrix(fmt, rec[2 * mgu:2 * mgu + mdn], H, I, g[2])
        x = _bf16_values(synth.hidden_ar1(11, 0, 0, 1, H, 0.9)[0])
        gv, uv = Wg @ x, Wu @ x
        want = Wd @ (gv / (1 + np.exp(-gv)) * uv)
        got = oracle.expert_ffn(fmt, rec, H, I, x)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-14 * np.abs(want).max()), fmt


def test_layer_is_weighted_sum_plus_shared():
    fmt, H, I, E, k = "bf16", 64, 32, 8, 3
    recs = {e: synth.expert_record(fmt, 5, 0, e, H, I) for e in range(E)}
    shared = synth.expert_record(fmt, 5, 0, -1, H, I)
    W = synth.router_weights(5, 0, E, H)
    b = synth.zipf_bias(E)
    x = synth.hidden_ar1(5, 0, 0, 3, H, 0.8)
    ids, wts, y = oracle.moe_layer(fmt, H, I, E, k, recs, x, W, b, shared=shared)
    z = oracle.router_logits(x, W, b)
    ids2, w2 = oracle.topk(z, k)
    assert np.array_equal(ids, ids2) and np.array_equal(wts, w2)
    for t in range(3):
        xt = _bf16_values(x[t])
        want = sum(wts[t, j] * oracle.expert_ffn(fmt, recs[ids[t, j]], H, I, xt) for j in range(k))
        want = want + oracle.expert_ffn(fmt, shared, H, I, xt)
        assert np.allclose(y[t], want, rtol=1e-13, atol=1e-16)
    # zero-weight mode: with the routed weights ignored only the shared FFN remains
    _, _, y_noshared = oracle.moe_layer(fmt, H, I, E, k, recs, x, W, b, shared=None)
    for t in range(3):
        xt = _bf16_values(x[t])
        assert np.allclose(y[t] - y_noshared[t], oracle.expert_ffn(fmt, shared, H, I, xt), rtol=1e-12, atol=1e-15)
