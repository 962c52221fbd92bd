"""The routing entry point that allocates nothing (moe_route_topk_noalloc).

It serves callers that cannot allocate device memory where they route
tokens (allocators that must not be re-entered from their own callbacks,
embedders that budget all device memory up front). Its ids must be exactly
those moe_layer_forward routes the same tokens to, and its weights those of
the oracle, on two calls in a row that share the library's fixed scratch
array. Collected last so a failure here does not hide the others.
"""
import numpy as np
import pytest

from harness import OracleRun, Setup, cuda_available
from synth.workloads import WORKLOADS, scaled

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


@pytest.mark.parametrize("name,T,H,norm", [("qwen3_30b_a3b_fp8", 4, 512, True), ("flash_next_nvfp4", 1, 512, True),
                                            ("tiny", 4, 256, True), ("qwen3_30b_a3b_q4_0", 3, 320, True),
                                            ("flash_next_nvfp4", 2, 512, False)])
def test_noalloc_routing_matches_the_layer_forward(name, T, H, norm):
    import torch
    import paged_expert_cache_gb300 as pec
    base = WORKLOADS[name]
    w = scaled(base, L=1, H=H, I=128, streams=(T,), steps=2,
               slots_per_layer=max(base.slots_per_layer, T * base.k), pool_bytes=0.0, pool_mode="per_layer",
               has_shared=False)
    st = Setup(w, max_tokens=T, norm_topk=norm)
    orc = OracleRun(w, st.info["slot_bytes"], norm=norm)
    xs = st.hiddens(0, T, 2)
    ids = torch.empty((T, w.k), dtype=torch.int32, device=st.dev)
    wts = torch.empty((T, w.k), dtype=torch.float32, device=st.dev)
    for step in range(2):  # two calls in a row share the scratch array
        st.forward(xs[step], 0)
        rec = st.cache.trace_read()[0]
        x = torch.from_numpy(np.ascontiguousarray(xs[step]).view(np.int16)).to(st.dev)
        pec.route_topk_noalloc(x, st.router_dev[0], ids, wts, w.k, bias=st.bias_dev, norm_topk=norm)
        torch.cuda.synchronize()
        got_ids = ids.cpu().numpy().reshape(-1)
        assert np.array_equal(got_ids, rec["ids"]), (got_ids, rec["ids"])
        want_ids, want_w = orc.route(xs[step], st.router[0], st.bias)
        assert np.array_equal(got_ids, want_ids.reshape(-1))
        assert np.allclose(wts.cpu().numpy(), want_w, rtol=1e-5, atol=1e-7)
    st.close()


def test_noalloc_refuses_sizes_beyond_its_scratch():
    import torch
    import paged_expert_cache_gb300 as pec
    dev = torch.device("cuda:0")
    x = torch.zeros((33, 256), dtype=torch.int16, device=dev)
    wr = torch.zeros((16, 256), dtype=torch.int16, device=dev)
    ids = torch.empty((33, 2), dtype=torch.int32, device=dev)
    wts = torch.empty((33, 2), dtype=torch.float32, device=dev)
    with pytest.raises(pec.MoeError) as ei:
        pec.route_topk_noalloc(x, wr, ids, wts, 2)
    assert ei.value.status == pec.ERR_INVALID
    wr_big = torch.zeros((513, 256), dtype=torch.int16, device=dev)
    with pytest.raises(pec.MoeError):
        pec.route_topk_noalloc(x[:1], wr_big, ids[:1], wts[:1], 2)
