"""Python binding of libmoecache.so, the C ABI declared in include/moe_cache.h.

Argument marshalling only: every step of the MoE layer (routing, the cache
plan, miss uploads, the expert FFN and the combine) runs in the library's
CUDA kernels. PyTorch is used by callers for device memory and streams; here
it only supplies data pointers and the current stream. There is no CPU
fallback: if the library is missing or fails to load, using it raises.
"""
import ctypes
import os
import re

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoecache.so")
HEADER = os.path.join(_HERE, "..", "include", "moe_cache.h")

OK, ERR_INVALID, ERR_CAPACITY, ERR_CUDA, ERR_OOM, ERR_STATE, ERR_TIMEOUT = range(7)
FORMATS = {"bf16": 0, "q4_0": 1, "fp8_b128": 2, "nvfp4": 3}
POOL_MODES = {"per_layer": 0, "shared": 1}
UPLOAD_MODES = {"pull": 0, "memcpy": 1}
DECODE_MODES = {"auto": 0, "three_kernels": 1, "one_kernel": 2}
EVICTIONS = {"lru": 0, "lfu": 1}
PREFILL_MODES = {"read_only": 0, "page_in": 1}
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID", 2: "MOE_ERR_CAPACITY", 3: "MOE_ERR_CUDA", 4: "MOE_ERR_OOM",
                5: "MOE_ERR_STATE", 6: "MOE_ERR_TIMEOUT"}

i32, u64, dbl, vp = ctypes.c_int32, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p


class MoeConfig(ctypes.Structure):
    _fields_ = [("num_layers", i32), ("num_experts", i32), ("top_k", i32), ("hidden", i32), ("inter", i32),
                ("format", i32), ("has_shared", i32), ("pool_mode", i32), ("slots_per_layer", i32),
                ("upload_mode", i32), ("pool_bytes", dbl), ("norm_topk", i32), ("max_cache_tokens", i32),
                ("prefill_group", i32), ("max_tokens", i32), ("device", i32), ("split_decode", i32),
                ("multi_wave", i32), ("eviction", i32), ("speculate", i32), ("prefill_mode", i32),
                ("adapt_period", i32), ("adapt_step", i32), ("adapt_min_slots", i32), ("adapt_max_slots", i32)]


class BucketStats(ctypes.Structure):
    _fields_ = [("calls", u64), ("hits", u64), ("misses", u64), ("bytes_uploaded", u64), ("upload_ns", u64)]


class MoeStats(ctypes.Structure):
    _fields_ = [("bucket", BucketStats * 3), ("num_pools", i32), ("slots_per_pool", i32), ("slot_bytes", u64),
                ("record_bytes", u64), ("topk_fp64_rerank", u64), ("spec_prefetched", u64), ("spec_used", u64)]


class MoeInfo(ctypes.Structure):
    _fields_ = [("num_pools", i32), ("slots_per_pool", i32), ("slot_bytes", u64), ("slot_stride", u64),
                ("record_bytes", u64), ("pool_device_bytes", u64), ("store_host_bytes", u64),
                ("scratch_device_bytes", u64), ("fused_decode_calls", u64), ("split_decode_calls", u64)]


NUM_STAGES = 7
STAGES = ["route", "copy", "gateup", "down", "prefill_topk", "prefill_plan", "layer"]


class MoeProfile(ctypes.Structure):
    _fields_ = [("ms", dbl * NUM_STAGES), ("launches", u64 * NUM_STAGES)]


_lib = None


def load():
    """Loads libmoecache.so (after torch, so both share one CUDA runtime)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() (nvcc, sm_103a) first")
    try:
        import torch  # noqa: F401  (loads the CUDA runtime torch uses)
    except ImportError:
        pass
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    sig = {
        "moe_config_default": (None, [P(MoeConfig)]),
        "moe_abi_version": (i32, []),
        "moe_last_error": (ctypes.c_char_p, [vp]),
        "moe_cache_create": (i32, [P(MoeConfig), vp, vp, P(vp)]),
        "moe_cache_load_experts": (i32, [vp, i32, i32, i32, vp]),
        "moe_cache_load_shared": (i32, [vp, i32, vp]),
        "moe_layer_forward": (i32, [vp, vp, i32, vp, vp, i32, vp, vp]),
        "moe_cache_stats": (i32, [vp, P(MoeStats)]),
        "moe_cache_info": (i32, [vp, P(MoeInfo)]),
        "moe_cache_trace_enable": (i32, [vp, i32]),
        "moe_cache_trace_read": (i32, [vp, vp, ctypes.c_int64, P(ctypes.c_int64), P(i32)]),
        "moe_cache_get_state": (i32, [vp, vp, vp, vp]),
        "moe_cache_read_slot": (i32, [vp, i32, i32, vp, i32, i32, vp, u64]),
        "moe_cache_profile_enable": (i32, [vp, i32]),
        "moe_cache_profile_read": (i32, [vp, P(MoeProfile)]),
        "moe_route_topk_noalloc": (i32, [vp, i32, vp, vp, i32, i32, i32, i32, vp, vp, vp]),
        "moe_cache_set_router": (i32, [vp, i32, vp, vp]),
        "moe_cache_pool_slots": (i32, [vp, vp]),
        "moe_cache_reset": (i32, [vp]),
        "moe_cache_destroy": (i32, [vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def header_functions():
    """Names of the entry points include/moe_cache.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


class MoeError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _check(st, handle=None):
    if st != OK:
        msg = load().moe_last_error(handle)
        raise MoeError(st, msg.decode() if msg else "")


def make_config(L, E, k, H, I, fmt="bf16", pool_mode="per_layer", slots_per_layer=0, pool_bytes=0.0,
                has_shared=False, upload_mode="pull", norm_topk=True, max_cache_tokens=32, prefill_group=32,
                max_tokens=32, device=0, decode="auto", multi_wave=False, eviction="lru", speculate=False,
                prefill="read_only", adapt=None):
    c = MoeConfig()
    load().moe_config_default(ctypes.byref(c))
    c.num_layers, c.num_experts, c.top_k, c.hidden, c.inter = L, E, k, H, I
    c.format = FORMATS[fmt] if isinstance(fmt, str) else int(fmt)
    c.pool_mode = POOL_MODES[pool_mode] if isinstance(pool_mode, str) else int(pool_mode)
    c.slots_per_layer = slots_per_layer
    c.pool_bytes = float(pool_bytes)
    c.has_shared = 1 if has_shared else 0
    c.upload_mode = UPLOAD_MODES[upload_mode] if isinstance(upload_mode, str) else int(upload_mode)
    c.norm_topk = 1 if norm_topk else 0
    c.max_cache_tokens = max_cache_tokens
    c.prefill_group = prefill_group
    c.max_tokens = max_tokens
    c.device = device
    c.split_decode = DECODE_MODES[decode] if isinstance(decode, str) else int(decode)
    c.multi_wave = 1 if multi_wave else 0
    c.eviction = EVICTIONS[eviction] if isinstance(eviction, str) else int(eviction)
    c.speculate = 1 if speculate else 0
    c.prefill_mode = PREFILL_MODES[prefill] if isinstance(prefill, str) else int(prefill)
    if adapt is not None:  # (period, step, min slots, max slots); 0 takes the default
        c.adapt_period, c.adapt_step, c.adapt_min_slots, c.adapt_max_slots = (int(v) for v in adapt)
    return c


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _refuse(msg):
    raise MoeError(ERR_INVALID, msg)


def _check_noalloc_args(hidden, router_w, ids, weights, top_k, bias):
    """Shapes, dtypes, devices and layouts of moe_route_topk_noalloc's tensors,
    checked before the C call: the kernel writes ids[t * k + j] and weights[t *
    k + j] for every token, so an undersized or mistyped output would be
    written out of bounds on the device."""
    import torch
    for name, t in (("hidden", hidden), ("router_w", router_w), ("ids", ids), ("weights", weights)):
        if not isinstance(t, torch.Tensor):
            _refuse(f"{name} must be a torch tensor")
    if hidden.dim() != 2 or router_w.dim() != 2:
        _refuse("hidden must be [T, H] and router_w [E, H]")
    T, H = hidden.shape
    E = router_w.shape[0]
    if router_w.shape[1] != H:
        _refuse(f"router_w has {router_w.shape[1]} columns, hidden has {H}")
    if hidden.element_size() != 2 or router_w.element_size() != 2:
        _refuse("hidden and router_w must hold 16-bit (bf16) values")
    if not isinstance(top_k, int) or top_k < 1:
        _refuse("top_k must be a positive int")
    if tuple(ids.shape) != (T, top_k) or ids.dtype != torch.int32:
        _refuse(f"ids must be int32 [{T}, {top_k}]")
    if tuple(weights.shape) != (T, top_k) or weights.dtype != torch.float32:
        _refuse(f"weights must be float32 [{T}, {top_k}]")
    tensors = [hidden, router_w, ids, weights]
    if bias is not None:
        if not isinstance(bias, torch.Tensor) or tuple(bias.shape) != (E,) or bias.dtype != torch.float32:
            _refuse(f"bias must be float32 [{E}]")
        tensors.append(bias)
    if not all(t.is_contiguous() for t in tensors):
        _refuse("every tensor must be contiguous")
    if not all(t.is_cuda for t in tensors):
        _refuse("every tensor must be on a CUDA device")
    dev = torch.cuda.current_device()
    if any(t.device.index != dev for t in tensors):
        _refuse(f"every tensor must be on the current CUDA device (cuda:{dev})")


def route_topk_noalloc(hidden, router_w, ids, weights, top_k, bias=None, norm_topk=True, stream=None):
    """moe_route_topk_noalloc: routing of T tokens into caller-provided ids
    [T, k] (int32) and weights [T, k] (fp32), with no allocation. The tensors
    are checked (shape, dtype, device, contiguity) before the call; a mismatch
    raises MoeError(ERR_INVALID) and launches nothing."""
    _check_noalloc_args(hidden, router_w, ids, weights, top_k, bias)
    T, H = hidden.shape
    E = router_w.shape[0]
    if stream is None:
        try:
            import torch
            stream = torch.cuda.current_stream().cuda_stream
        except Exception:
            stream = 0
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    _check(load().moe_route_topk_noalloc(_ptr(hidden), T, _ptr(router_w), _ptr(bias), E, H, top_k,
                                         1 if norm_topk else 0, _ptr(ids), _ptr(weights), stream or None))
    return ids, weights


class MoECache:
    """One handle of the C library (moe_cache_t*)."""

    def __init__(self, cfg, expert_host=None, shared_host=None):
        L = load()
        self.cfg = cfg
        h = vp()
        eh = sh = None
        if expert_host is not None:
            arr = (vp * cfg.num_layers)(*[_ptr(a) for a in expert_host])
            eh = ctypes.cast(arr, vp)
        if shared_host is not None:
            arr2 = (vp * cfg.num_layers)(*[_ptr(a) for a in shared_host])
            sh = ctypes.cast(arr2, vp)
        _check(L.moe_cache_create(ctypes.byref(cfg), eh, sh, ctypes.byref(h)))
        self.h = h.value

    def close(self):
        if getattr(self, "h", None):
            load().moe_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_experts(self, layer, first, records):
        records = np.ascontiguousarray(records, dtype=np.uint8)
        n = records.shape[0] if records.ndim == 2 else 1
        _check(load().moe_cache_load_experts(self.h, layer, first, n, records.ctypes.data), self.h)

    def load_shared(self, layer, record):
        record = np.ascontiguousarray(record, dtype=np.uint8)
        _check(load().moe_cache_load_shared(self.h, layer, record.ctypes.data), self.h)

    def forward(self, hidden, router_w, layer, out, bias=None, stream=None, T=None):
        """hidden: device bf16 [T, H]; router_w: device bf16 [E, H]; bias:
        device fp32 [E] or None; out: device fp32 [T, H]. Pointers (ints) or
        tensors. stream: a cudaStream_t as int, a torch stream, or None for
        torch's current stream."""
        if T is None:
            T = hidden.shape[0]
        if stream is None:
            try:
                import torch
                stream = torch.cuda.current_stream().cuda_stream
            except Exception:
                stream = 0
        elif not isinstance(stream, int):
            stream = stream.cuda_stream
        _check(load().moe_layer_forward(self.h, _ptr(hidden), T, _ptr(router_w), _ptr(bias), layer, _ptr(out),
                                        stream or None), self.h)
        return out

    def set_router(self, layer, router_w, bias=None):
        """moe_cache_set_router: registers layer's router (device bf16 [E, H],
        device fp32 [E] or None) for speculative next-layer routing; the
        tensors must stay alive and unchanged while registered."""
        _check(load().moe_cache_set_router(self.h, layer, _ptr(router_w), _ptr(bias)), self.h)

    def pool_slots(self):
        """moe_cache_pool_slots: the slots each pool holds now."""
        n = self.info()["num_pools"]
        out = np.empty(n, dtype=np.int32)
        _check(load().moe_cache_pool_slots(self.h, out.ctypes.data), self.h)
        return out.tolist()

    def stats(self):
        s = MoeStats()
        _check(load().moe_cache_stats(self.h, ctypes.byref(s)), self.h)
        buckets = [{f: getattr(s.bucket[b], f) for f, _ in BucketStats._fields_} for b in range(3)]
        return {"buckets": buckets, "num_pools": s.num_pools, "slots_per_pool": s.slots_per_pool,
                "slot_bytes": s.slot_bytes, "record_bytes": s.record_bytes, "topk_fp64_rerank": s.topk_fp64_rerank,
                "spec_prefetched": s.spec_prefetched, "spec_used": s.spec_used}

    def info(self):
        s = MoeInfo()
        _check(load().moe_cache_info(self.h, ctypes.byref(s)), self.h)
        return {f: getattr(s, f) for f, _ in MoeInfo._fields_}

    def trace_enable(self, capacity):
        _check(load().moe_cache_trace_enable(self.h, capacity), self.h)

    def trace_read(self, max_words=1 << 24):
        buf = np.empty(max_words, dtype=np.int32)
        nw, nr = ctypes.c_int64(0), i32(0)
        _check(load().moe_cache_trace_read(self.h, buf.ctypes.data, max_words, ctypes.byref(nw), ctypes.byref(nr)),
               self.h)
        out, p = [], 0
        for _ in range(nr.value):
            layer, T, ni, nh, nf, nu = (int(v) for v in buf[p:p + 6])
            p += 6
            rec = {"layer": layer, "T": T, "n_hit": nh, "n_fill": nf, "n_uniq": nu}
            rec["ids"] = buf[p:p + ni].copy(); p += ni
            rec["slot_of"] = buf[p:p + ni].copy(); p += ni
            rec["hit_of"] = buf[p:p + ni].copy(); p += ni
            rec["fill_expert"] = buf[p:p + nf].copy(); p += nf
            rec["fill_slot"] = buf[p:p + nf].copy(); p += nf
            out.append(rec)
        return out

    def state(self):
        c = self.cfg
        info = self.info()
        npools, K = info["num_pools"], info["slots_per_pool"]
        sm = np.empty(c.num_layers * c.num_experts, dtype=np.int32)
        ko = np.empty(npools * K, dtype=np.int32)
        order = np.empty(npools * K, dtype=np.int32)
        _check(load().moe_cache_get_state(self.h, sm.ctypes.data, ko.ctypes.data, order.ctypes.data), self.h)
        return {"slot_map": sm.reshape(c.num_layers, c.num_experts), "key_of": ko.reshape(npools, K),
                "order": order.reshape(npools, K)}

    def read_slot(self, pool, slot, layer=-1, expert=-1, nbytes=None):
        """(slot bytes on the device, the store's bytes of (layer, expert) or None)."""
        if nbytes is None:
            nbytes = self.info()["slot_bytes"]
        dst = np.empty(nbytes, dtype=np.uint8)
        store = np.empty(nbytes, dtype=np.uint8) if layer >= 0 else None
        _check(load().moe_cache_read_slot(self.h, pool, slot, dst.ctypes.data, layer, expert,
                                          None if store is None else store.ctypes.data, nbytes), self.h)
        return dst, store

    def profile_enable(self, on=True):
        _check(load().moe_cache_profile_enable(self.h, 1 if on else 0), self.h)

    def profile_read(self):
        p = MoeProfile()
        _check(load().moe_cache_profile_read(self.h, ctypes.byref(p)), self.h)
        return {STAGES[i]: {"ms": p.ms[i], "launches": p.launches[i]} for i in range(NUM_STAGES)}

    def reset(self):
        _check(load().moe_cache_reset(self.h), self.h)
