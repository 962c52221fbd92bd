"""Python marshalling for the CPU oracle (liboracle.so built from moe_oracle.c).

TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import this package; the product path never
does. Every computation happens in moe_oracle.c (plain fp64 C); this file
only converts numpy arrays to pointers and back.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_SO = os.path.join(_HERE, "liboracle.so")

FMT = {"bf16": 0, "q4_0": 1, "fp8_b128": 2, "nvfp4": 3}
POOL = {"per_layer": 0, "shared": 1}
POLICY = {"lru": 0, "lfu": 1}
PREFILL = {"read_only": 0, "page_in": 1}
OK, ERR_INVALID, ERR_CAPACITY, ERR_MISSING = 0, 1, 2, 3

_lib = None


def build(force=False):
    """Compile liboracle.so: portable C11, fp64, no fused multiply-adds."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest:
        return _SO
    tmp = _SO + ".tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        i32, dbl, vp, sz = ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_size_t
        L.orc_decode_fp16.restype = dbl
        L.orc_decode_fp16.argtypes = [ctypes.c_uint16]
        L.orc_decode_bf16.restype = dbl
        L.orc_decode_bf16.argtypes = [ctypes.c_uint16]
        L.orc_decode_e4m3.restype = dbl
        L.orc_decode_e4m3.argtypes = [ctypes.c_uint8]
        L.orc_decode_e2m1.restype = dbl
        L.orc_decode_e2m1.argtypes = [ctypes.c_uint8]
        L.orc_decode_array.argtypes = [i32, vp, sz, vp]
        L.orc_matrix_bytes.restype = sz
        L.orc_matrix_bytes.argtypes = [i32, i32, i32]
        L.orc_record_bytes.restype = sz
        L.orc_record_bytes.argtypes = [i32, i32, i32]
        L.orc_slot_bytes.restype = sz
        L.orc_slot_bytes.argtypes = [i32, i32, i32]
        L.orc_slots_for_budget.restype = ctypes.c_int64
        L.orc_slots_for_budget.argtypes = [dbl, dbl]
        L.orc_dequant_matrix.argtypes = [i32, vp, i32, i32, dbl, vp]
        L.orc_router_logits.argtypes = [vp, i32, i32, vp, i32, vp, vp]
        L.orc_topk.argtypes = [vp, i32, i32, i32, i32, vp, vp]
        L.orc_expert_ffn.argtypes = [i32, vp, i32, i32, vp, vp]
        L.orc_moe_layer.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp]
        L.orc_cache_create.restype = vp
        L.orc_cache_create.argtypes = [i32, i32, i32, i32, dbl, i32]
        L.orc_cache_destroy.argtypes = [vp]
        L.orc_cache_reset.argtypes = [vp]
        L.orc_cache_plan.argtypes = [vp, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        L.orc_cache_state.argtypes = [vp, vp, vp, vp]
        L.orc_cache_num_pools.argtypes = [vp]
        L.orc_cache_slots.argtypes = [vp]
        L.orc_cache_stats.argtypes = [vp, vp]
        L.orc_count_runs.argtypes = [vp, vp, i32]
        L.orc_wave_split.argtypes = [i32, i32, i32, vp, vp]
        L.orc_cache_set_policy.argtypes = [vp, i32]
        L.orc_cache_set_prefill_mode.argtypes = [vp, i32]
        L.orc_cache_set_adaptive.argtypes = [vp, i32, i32, i32, i32]
        L.orc_cache_pool_slots.argtypes = [vp, i32]
        _lib = L
    return _lib


def _fmt(f):
    return FMT[f] if isinstance(f, str) else int(f)


def _p(a):
    return None if a is None else a.ctypes.data


def decode(kind, codes):
    """kind in {'fp16','bf16','e4m3','e2m1'}: codes -> float64 via the oracle."""
    k = {"fp16": 0, "bf16": 1, "e4m3": 2, "e2m1": 3}[kind]
    a = np.ascontiguousarray(codes, dtype=np.uint16 if k < 2 else np.uint8)
    out = np.empty(a.size, dtype=np.float64)
    assert lib().orc_decode_array(k, a.ctypes.data, a.size, out.ctypes.data) == OK
    return out.reshape(a.shape)


def matrix_bytes(fmt, rows, cols):
    return int(lib().orc_matrix_bytes(_fmt(fmt), rows, cols))


def record_bytes(fmt, H, I):
    return int(lib().orc_record_bytes(_fmt(fmt), H, I))


def slot_bytes(fmt, H, I):
    return int(lib().orc_slot_bytes(_fmt(fmt), H, I))


def slots_for_budget(pool_bytes, per_slot_bytes):
    return int(lib().orc_slots_for_budget(float(pool_bytes), float(per_slot_bytes)))


def dequant_matrix(fmt, mat, rows, cols, g=1.0):
    m = np.ascontiguousarray(mat, dtype=np.uint8)
    out = np.empty((rows, cols), dtype=np.float64)
    assert lib().orc_dequant_matrix(_fmt(fmt), m.ctypes.data, rows, cols, float(g), out.ctypes.data) == OK
    return out


def router_logits(x_bf16, w_bf16, bias=None):
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    T, H = x.shape
    E = w.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    z = np.empty((T, E), dtype=np.float64)
    lib().orc_router_logits(x.ctypes.data, T, H, w.ctypes.data, E, _p(b), z.ctypes.data)
    return z


def topk(z, k, norm=True):
    z = np.ascontiguousarray(z, dtype=np.float64)
    T, E = z.shape
    ids = np.empty((T, k), dtype=np.int32)
    wts = np.empty((T, k), dtype=np.float64)
    lib().orc_topk(z.ctypes.data, T, E, k, 1 if norm else 0, ids.ctypes.data, wts.ctypes.data)
    return ids, wts


def expert_ffn(fmt, record, H, I, x):
    r = np.ascontiguousarray(record, dtype=np.uint8)
    xv = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(H, dtype=np.float64)
    assert lib().orc_expert_ffn(_fmt(fmt), r.ctypes.data, H, I, xv.ctypes.data, y.ctypes.data) == OK
    return y


def moe_layer(fmt, H, I, E, k, records, x_bf16, router_w, bias=None, shared=None, norm=True):
    """The unpaged layer. records: mapping expert -> uint8 record (only the
    selected experts are needed). Returns ids [T,k], wts [T,k], y [T,H] fp64."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    w = np.ascontiguousarray(router_w, dtype=np.uint16)
    T = x.shape[0]
    keep = [None] * E
    ptrs = (ctypes.c_void_p * E)()
    for e, r in (records.items() if isinstance(records, dict) else enumerate(records)):
        if r is None:
            continue
        keep[e] = np.ascontiguousarray(r, dtype=np.uint8)
        ptrs[e] = keep[e].ctypes.data
    sh = None if shared is None else np.ascontiguousarray(shared, dtype=np.uint8)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    ids = np.empty((T, k), dtype=np.int32)
    wts = np.empty((T, k), dtype=np.float64)
    y = np.empty((T, H), dtype=np.float64)
    rc = lib().orc_moe_layer(_fmt(fmt), H, I, E, k, 1 if norm else 0, ctypes.cast(ptrs, ctypes.c_void_p),
                             _p(sh), x.ctypes.data, T, w.ctypes.data, _p(b), ids.ctypes.data,
                             wts.ctypes.data, y.ctypes.data)
    if rc != OK:
        raise RuntimeError(f"orc_moe_layer failed: {rc}")
    return ids, wts, y


def count_runs(fill_expert, fill_slot):
    fe = np.ascontiguousarray(fill_expert, dtype=np.int32)
    fs = np.ascontiguousarray(fill_slot, dtype=np.int32)
    return int(lib().orc_count_runs(fe.ctypes.data, fs.ctypes.data, fe.size))


def wave_split(T, k, K):
    """[(first token, tokens)] of each wave of a decode step (moe_oracle.c)."""
    start = np.empty(max(T, 1), dtype=np.int32)
    count = np.empty(max(T, 1), dtype=np.int32)
    n = int(lib().orc_wave_split(T, k, K, start.ctypes.data, count.ctypes.data))
    return [(int(start[i]), int(count[i])) for i in range(n)]


class CacheError(RuntimeError):
    def __init__(self, code):
        super().__init__(f"oracle cache error {code}")
        self.code = code


class Cache:
    """The literal LRU list (moe_oracle.c), one instance per simulated cache."""

    def __init__(self, L, E, pool_mode, slots_per_pool, slot_bytes=0.0, max_cache_tokens=32, policy="lru",
                 prefill="read_only", adaptive=None):
        self.L, self.E = L, E
        self.h = lib().orc_cache_create(L, E, POOL[pool_mode] if isinstance(pool_mode, str) else pool_mode,
                                        slots_per_pool, float(slot_bytes), max_cache_tokens)
        if not self.h:
            raise ValueError("invalid oracle cache configuration")
        if lib().orc_cache_set_policy(self.h, POLICY.get(policy, -1)) != OK:
            raise ValueError("invalid eviction policy")
        if lib().orc_cache_set_prefill_mode(self.h, PREFILL.get(prefill, -1)) != OK:
            raise ValueError("invalid prefill mode")
        if adaptive is not None:  # (period, step, kmin, kmax)
            if lib().orc_cache_set_adaptive(self.h, *[int(v) for v in adaptive]) != OK:
                raise ValueError("invalid adaptive capacity")
        self.n_pools = lib().orc_cache_num_pools(self.h)
        self.K = lib().orc_cache_slots(self.h)

    def pool_slots(self):
        """Slots each pool holds now (the configured K unless capacity adapts)."""
        return [int(lib().orc_cache_pool_slots(self.h, p)) for p in range(self.n_pools)]

    def __del__(self):
        h = getattr(self, "h", None)
        if h and _lib is not None:
            _lib.orc_cache_destroy(h)
            self.h = None

    def reset(self):
        lib().orc_cache_reset(self.h)

    def plan(self, layer, ids, T=None):
        ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
        n = ids.size
        if T is None:
            T = 1
        slot_of = np.empty(n, dtype=np.int32)
        hit_of = np.empty(n, dtype=np.uint8)
        fe = np.empty(max(n, 1), dtype=np.int32)
        fs = np.empty(max(n, 1), dtype=np.int32)
        nf, nh, nu = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
        rc = lib().orc_cache_plan(self.h, layer, ids.ctypes.data, n, T, slot_of.ctypes.data,
                                  hit_of.ctypes.data, fe.ctypes.data, fs.ctypes.data,
                                  ctypes.byref(nf), ctypes.byref(nh), ctypes.byref(nu))
        if rc != OK:
            raise CacheError(rc)
        return {"slot_of": slot_of, "hit_of": hit_of, "fill_expert": fe[:nf.value].copy(),
                "fill_slot": fs[:nf.value].copy(), "n_hit": nh.value, "n_uniq": nu.value,
                "n_fill": nf.value}

    def state(self):
        sm = np.empty(self.L * self.E, dtype=np.int32)
        ko = np.empty(self.n_pools * self.K, dtype=np.int32)
        order = np.empty(self.n_pools * self.K, dtype=np.int32)
        lib().orc_cache_state(self.h, sm.ctypes.data, ko.ctypes.data, order.ctypes.data)
        return {"slot_map": sm.reshape(self.L, self.E), "key_of": ko.reshape(self.n_pools, self.K),
                "order": order.reshape(self.n_pools, self.K)}

    def stats(self):
        s = np.empty(12, dtype=np.uint64)
        lib().orc_cache_stats(self.h, s.ctypes.data)
        s = s.reshape(3, 4)
        return [{"calls": int(r[0]), "hits": int(r[1]), "misses": int(r[2]), "bytes": int(r[3])} for r in s]
