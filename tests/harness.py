"""Shared helpers for the GPU parity tests: build a cache from a synthetic
workload, run decode steps through the C ABI, and run the same steps through
the oracle (test infrastructure only)."""
import numpy as np

import oracle
import synth


def cuda_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def rel_l2(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def pool_slots(w, slot_bytes, K=None):
    if w.pool_mode == "per_layer":
        return K if K is not None else w.slots_per_layer
    return oracle.slots_for_budget(w.pool_bytes, slot_bytes)


class Setup:
    """A GPU cache plus the workload's device inputs."""

    def __init__(self, w, K=None, upload="pull", max_tokens=None, pool_bytes=None, trace=4096, decode="auto",
                 multi_wave=False, eviction="lru", norm_topk=True, speculate=False, prefill="read_only",
                 adapt=None):
        import torch
        import paged_expert_cache_gb300 as pec
        self.w = w
        mt = max_tokens or max(max(w.streams), w.prompt_T or 0)
        cfg = pec.make_config(w.L, w.E, w.k, w.H, w.I, fmt=w.fmt, pool_mode=w.pool_mode,
                              slots_per_layer=(K if K is not None else w.slots_per_layer),
                              pool_bytes=(pool_bytes if pool_bytes is not None else w.pool_bytes),
                              has_shared=w.has_shared, upload_mode=upload, max_tokens=mt,
                              decode=decode, multi_wave=multi_wave, eviction=eviction, norm_topk=norm_topk,
                              speculate=speculate, prefill=prefill, adapt=adapt)
        self.cache = pec.MoECache(cfg)
        buf = None
        for l in range(w.L):
            buf = synth.expert_records(w.fmt, w.seed, l, 0, w.E, w.H, w.I, out=buf)
            self.cache.load_experts(l, 0, buf)
            if w.has_shared:
                self.cache.load_shared(l, synth.expert_record(w.fmt, w.seed, l, -1, w.H, w.I))
        if trace:
            self.cache.trace_enable(trace)
        self.info = self.cache.info()
        self.router = [synth.router_weights(w.seed, l, w.E, w.H) for l in range(w.L)]
        self.bias = synth.zipf_bias(w.E) if w.bias else None
        dev = torch.device("cuda:0")
        self.router_dev = [torch.from_numpy(r.view(np.int16)).to(dev) for r in self.router]
        self.bias_dev = None if self.bias is None else torch.from_numpy(self.bias).to(dev)
        self.dev = dev
        if speculate:
            for l in range(w.L):
                self.cache.set_router(l, self.router_dev[l], self.bias_dev)

    def hiddens(self, layer, T, steps, rho=None):
        """[steps, T, H] bf16 bits: T independent AR(1) streams."""
        w = self.w
        seq = [synth.hidden_ar1(w.seed, layer, s, steps, w.H, w.rho if rho is None else rho) for s in range(T)]
        return np.stack(seq, axis=1)

    def forward(self, x_bits, layer):
        import torch
        T = x_bits.shape[0]
        x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(self.dev)
        out = torch.empty((T, self.w.H), dtype=torch.float32, device=self.dev)
        self.cache.forward(x, self.router_dev[layer], layer, out, bias=self.bias_dev)
        return out.cpu().numpy().astype(np.float64)

    def close(self):
        self.cache.close()


class OracleRun:
    """The same calls through the oracle: routing, literal LRU, unpaged layer."""

    def __init__(self, w, slot_bytes, K=None, policy="lru", norm=True, prefill="read_only", adaptive=None):
        self.w = w
        self.norm = norm
        self.K = pool_slots(w, slot_bytes, K)
        self.cache = oracle.Cache(w.L, w.E, w.pool_mode, self.K, slot_bytes, policy=policy, prefill=prefill,
                                  adaptive=adaptive)
        self._rec = {}

    def record(self, layer, e):
        key = (layer, e)
        if key not in self._rec:
            self._rec[key] = synth.expert_record(self.w.fmt, self.w.seed, layer, e, self.w.H, self.w.I)
        return self._rec[key]

    def route(self, x_bits, router, bias):
        z = oracle.router_logits(x_bits, router, bias)
        return oracle.topk(z, self.w.k, norm=self.norm)

    def plan(self, layer, ids, T):
        return self.cache.plan(layer, ids.reshape(-1), T)

    def layer(self, x_bits, router, bias, layer):
        w = self.w
        z = oracle.router_logits(x_bits, router, bias)
        ids, _ = oracle.topk(z, w.k)
        recs = {int(e): self.record(layer, int(e)) for e in np.unique(ids)}
        shared = self.record(layer, -1) if w.has_shared else None
        return oracle.moe_layer(w.fmt, w.H, w.I, w.E, w.k, recs, x_bits, router, bias, shared=shared,
                                norm=self.norm)


def compare_trace(rec, ids, plan, layer, T):
    """GPU trace record vs the oracle's routing and plan of the same call."""
    assert rec["layer"] == layer and rec["T"] == T
    assert np.array_equal(rec["ids"], ids.reshape(-1)), (rec["ids"], ids.reshape(-1))
    assert np.array_equal(rec["slot_of"], plan["slot_of"]), (rec["slot_of"], plan["slot_of"])
    assert np.array_equal(rec["hit_of"].astype(np.uint8), plan["hit_of"])
    assert np.array_equal(rec["fill_expert"], plan["fill_expert"])
    assert np.array_equal(rec["fill_slot"], plan["fill_slot"])
    assert rec["n_hit"] == plan["n_hit"] and rec["n_uniq"] == plan["n_uniq"]


def scale_bf16_rows(x_bits, factors):
    """bf16 bit patterns [T, H] with row t multiplied by factors[t] (or by an
    array broadcast against the row), rounded to nearest even: token rows of a
    chosen magnitude, built on the test side as inputs."""
    x = (np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    f = np.asarray(factors, dtype=np.float64)
    y = (x * (f[:, None] if f.ndim == 1 else f)).astype(np.float32)
    u = y.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def rel_l2_rows(got, want):
    """Relative L2 error of each row (token) separately."""
    return [rel_l2(g, w) for g, w in zip(np.asarray(got), np.asarray(want))]
