"""The C-ABI library loads, exports every entry point its header declares, and
validates configurations on the host (no GPU needed)."""
import ctypes

import pytest

import paged_expert_cache_gb300 as pec


def test_library_exports_every_header_function():
    lib = pec.load()
    names = pec.header_functions()
    assert "moe_layer_forward" in names and "moe_cache_create" in names and "moe_cache_stats" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert lib.moe_abi_version() == 3


def test_config_defaults():
    c = pec.MoeConfig()
    pec.load().moe_config_default(ctypes.byref(c))
    assert c.norm_topk == 1 and c.max_cache_tokens == 32 and c.prefill_group == 32 and c.max_tokens == 32
    assert c.upload_mode == 0 and c.pool_mode == 0
    assert c.split_decode == 0  # automatic choice of the decode launch
    assert c.multi_wave == 0  # single-wave rule: over-capacity decode calls are refused
    assert c.eviction == 0  # least recently used
    assert c.speculate == 0  # no speculative next-layer prefetch
    assert c.prefill_mode == 0  # prefill reads the cache without changing it
    assert c.adapt_period == 0  # fixed per-layer capacity


@pytest.mark.parametrize("kw,status", [
    (dict(L=0, E=16, k=2, H=256, I=128), pec.ERR_INVALID),
    (dict(L=1, E=2000, k=2, H=256, I=128), pec.ERR_INVALID),
    (dict(L=1, E=16, k=17, H=256, I=128), pec.ERR_INVALID),
    (dict(L=1, E=16, k=2, H=100, I=128), pec.ERR_INVALID),
    (dict(L=1, E=16, k=2, H=256, I=96), pec.ERR_INVALID),
    (dict(L=1, E=16, k=2, H=256, I=128, fmt=7), pec.ERR_INVALID),
    (dict(L=1, E=16, k=4, H=256, I=128, slots_per_layer=3), pec.ERR_CAPACITY),
    (dict(L=1, E=16, k=2, H=256, I=128, pool_mode="shared", pool_bytes=196608 * 2 - 1), pec.ERR_CAPACITY),
    (dict(L=1, E=16, k=2, H=256, I=128, slots_per_layer=8, max_cache_tokens=33), pec.ERR_INVALID),
    (dict(L=1, E=16, k=2, H=256, I=128, slots_per_layer=8, decode=3), pec.ERR_INVALID),
    (dict(L=1, E=16, k=2, H=256, I=128, slots_per_layer=8, eviction=2), pec.ERR_INVALID),
    (dict(L=1, E=16, k=2, H=256, I=128, slots_per_layer=8, speculate=True, upload_mode="memcpy"), pec.ERR_INVALID),
    (dict(L=1, E=16, k=2, H=256, I=128, slots_per_layer=8, prefill=2), pec.ERR_INVALID),
    (dict(L=2, E=16, k=2, H=256, I=128, pool_mode="shared", pool_bytes=196608 * 8, adapt=(1, 1, 0, 0)),
     pec.ERR_INVALID),
    (dict(L=2, E=16, k=2, H=256, I=128, slots_per_layer=8, adapt=(1, 1, 9, 12)), pec.ERR_INVALID),
    (dict(L=2, E=16, k=4, H=256, I=128, slots_per_layer=8, adapt=(1, 1, 3, 12)), pec.ERR_INVALID),
    (dict(L=1, E=16, k=2, H=256, I=128, slots_per_layer=8, prefill="page_in", eviction="lfu"), pec.ERR_INVALID),
])
def test_invalid_configurations_are_refused(kw, status):
    args = dict(kw)
    L, E, k, H, I = (args.pop(x) for x in ("L", "E", "k", "H", "I"))
    cfg = pec.make_config(L, E, k, H, I, **args)
    with pytest.raises(pec.MoeError) as ei:
        pec.MoECache(cfg)
    assert ei.value.status == status
    assert str(ei.value)


def test_multi_wave_flag_must_be_0_or_1():
    cfg = pec.make_config(1, 16, 2, 256, 128, slots_per_layer=8)
    cfg.multi_wave = 2
    with pytest.raises(pec.MoeError) as ei:
        pec.MoECache(cfg)
    assert ei.value.status == pec.ERR_INVALID


def test_noalloc_wrapper_refuses_mismatched_tensors_before_any_launch():
    # The routing entry point writes ids[t * k + j] and weights[t * k + j] for
    # every token: the binding refuses outputs of the wrong shape or dtype,
    # inputs whose widths differ, and non-contiguous tensors before it calls
    # the library (these CPU tensors never reach a kernel).
    torch = pytest.importorskip("torch")
    x = torch.zeros((4, 256), dtype=torch.int16)
    wr = torch.zeros((16, 256), dtype=torch.int16)
    ids = torch.zeros((4, 2), dtype=torch.int32)
    wts = torch.zeros((4, 2), dtype=torch.float32)
    bad = [
        (x, wr, torch.zeros((3, 2), dtype=torch.int32), wts, None, "ids"),
        (x, wr, torch.zeros((4, 2), dtype=torch.int64), wts, None, "ids"),
        (x, wr, ids, torch.zeros((4, 1), dtype=torch.float32), None, "weights"),
        (x, wr, ids, torch.zeros((4, 2), dtype=torch.float64), None, "weights"),
        (x, torch.zeros((16, 192), dtype=torch.int16), ids, wts, None, "columns"),
        (x.float(), wr, ids, wts, None, "16-bit"),
        (x, wr, ids, wts, torch.zeros(15, dtype=torch.float32), "bias"),
        (x, wr, torch.zeros((2, 4), dtype=torch.int32).t(), wts, None, "contiguous"),
        (x, wr, ids, wts, None, "CUDA device"),
    ]
    for h, r, i, w, b, what in bad:
        with pytest.raises(pec.MoeError) as ei:
            pec.route_topk_noalloc(h, r, i, w, 2, bias=b)
        assert ei.value.status == pec.ERR_INVALID
        assert what in str(ei.value), (what, str(ei.value))
