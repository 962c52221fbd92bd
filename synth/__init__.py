"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

Expert records in the four canonical weight formats, router weights, router
bias and hidden states. This package draws numbers and lays them out; it holds
none of the MoE method's arithmetic (no weight is decoded and no layer is
computed here). Every value is a pure function of its seed and coordinates,
so a record can be regenerated alone, e.g. to check a sampled output.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")

FORMATS = {"bf16": 0, "q4_0": 1, "fp8_b128": 2, "nvfp4": 3}

_lib = None


def build(force=False):
    """Compile libsynth.so with the host C compiler (portable C, no ISA flags)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + ".tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        u64, i32, dbl, vp, sz = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_size_t
        L.syn_key.restype = u64
        L.syn_key.argtypes = [u64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
        L.syn_normal_bf16.argtypes = [u64, sz, dbl, vp]
        L.syn_router_weights.argtypes = [u64, i32, i32, i32, dbl, vp]
        L.syn_prompt.argtypes = [u64, i32, i32, i32, dbl, vp]
        L.syn_hidden_ar1.argtypes = [u64, i32, i32, i32, i32, dbl, vp]
        L.syn_record_bytes.restype = sz
        L.syn_record_bytes.argtypes = [i32, i32, i32]
        L.syn_expert_record.argtypes = [i32, u64, i32, i32, i32, i32, vp]
        L.syn_expert_records.argtypes = [i32, u64, i32, i32, i32, i32, i32, vp, i32]
        _lib = L
    return _lib


def fmt_code(fmt):
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def record_bytes(fmt, H, I):
    """Canonical record bytes (NVFP4 includes its three fp32 global scales)."""
    return int(lib().syn_record_bytes(fmt_code(fmt), H, I))


def expert_record(fmt, seed, layer, expert, H, I):
    """One canonical record as uint8; expert=-1 is the layer's shared expert."""
    out = np.empty(record_bytes(fmt, H, I), dtype=np.uint8)
    lib().syn_expert_record(fmt_code(fmt), seed, layer, expert, H, I, out.ctypes.data)
    return out


def expert_records(fmt, seed, layer, e0, n, H, I, out=None, nthreads=None):
    """Records of experts e0..e0+n-1 of one layer as a [n, record_bytes] array."""
    rb = record_bytes(fmt, H, I)
    if out is None:
        out = np.empty((n, rb), dtype=np.uint8)
    assert out.dtype == np.uint8 and out.flags.c_contiguous and out.size >= n * rb
    nt = nthreads or min(16, os.cpu_count() or 1)
    lib().syn_expert_records(fmt_code(fmt), seed, layer, e0, n, H, I, out.ctypes.data, nt)
    return out


def router_weights(seed, layer, E, H, sd=0.02):
    """Router matrix [E, H] as bf16 bits (uint16), entries ~ N(0, sd)."""
    out = np.empty((E, H), dtype=np.uint16)
    lib().syn_router_weights(seed, layer, E, H, sd, out.ctypes.data)
    return out


def prompt(seed, layer, T, H, sd=1.0):
    """Prompt hiddens [T, H] as bf16 bits, i.i.d. N(0, sd) per layer."""
    out = np.empty((T, H), dtype=np.uint16)
    lib().syn_prompt(seed, layer, T, H, sd, out.ctypes.data)
    return out


def hidden_ar1(seed, layer, stream, nsteps, H, rho):
    """Decode hiddens [nsteps, H] (bf16 bits) of one stream: AR(1) with
    standard-normal innovations and correlation rho between steps."""
    out = np.empty((nsteps, H), dtype=np.uint16)
    lib().syn_hidden_ar1(seed, layer, stream, nsteps, H, rho, out.ctypes.data)
    return out


def zipf_bias(E, s=1.1, scale=0.5):
    """Per-expert router bias scale*(e+1)^-s: popular experts have low ids."""
    return (scale * np.power(np.arange(1, E + 1, dtype=np.float64), -s)).astype(np.float32)

