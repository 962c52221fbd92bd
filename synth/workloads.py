"""The five synthetic workloads, as plain data (shapes, seeds, input recipe).

Each stands in for a page's workload: the real checkpoints (Qwen3-30B-A3B,
Qwen3.8-Flash-Next) and prompt sets are not available, so inputs are seeded
draws with the same shapes. Nothing here computes any part of the method.
"""
from dataclasses import dataclass, field
from typing import Optional, Tuple

MASTER_SEED = 20261202


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    L: int            # MoE layers
    E: int            # routed experts per layer
    k: int            # top_k
    H: int            # hidden size
    I: int            # expert intermediate size
    fmt: str          # bf16 | q4_0 | fp8_b128 | nvfp4
    pool_mode: str    # per_layer | shared
    slots_per_layer: int = 0      # per-layer pools
    pool_bytes: float = 0.0       # shared pool
    has_shared: bool = False
    bias: bool = False            # Zipf(1.1)*0.5 router bias
    streams: Tuple[int, ...] = (1,)  # tokens per call (independent AR(1) streams)
    steps: int = 64
    rho: float = 0.9
    prompt_T: int = 0             # prefill prompt length (0 = none)
    note: str = ""

    @property
    def seed(self):
        return MASTER_SEED + self.index


WORKLOADS = {
    "tiny": Workload(
        name="tiny", index=1, L=1, E=16, k=2, H=256, I=128, fmt="bf16", pool_mode="per_layer",
        slots_per_layer=8, bias=True, streams=(4,), steps=64, rho=0.8,
        note="1 layer, 16 experts top-2, bf16, K=8 (= tokens*k: the capacity edge)"),
    "qwen3_30b_a3b_q4_0": Workload(
        name="qwen3_30b_a3b_q4_0", index=2, L=48, E=128, k=8, H=2048, I=768, fmt="q4_0",
        pool_mode="per_layer", slots_per_layer=92, bias=False, streams=(1,), steps=256, rho=0.9,
        note="Qwen3-30B-A3B-shaped decode, Q4_0 experts, 92 slots per layer, batch 1"),
    "qwen3_30b_a3b_fp8": Workload(
        name="qwen3_30b_a3b_fp8", index=3, L=48, E=128, k=8, H=2048, I=768, fmt="fp8_b128",
        pool_mode="per_layer", slots_per_layer=92, bias=True, streams=(1, 2, 4, 8), steps=256, rho=0.9,
        note="same shape, block-FP8 e4m3 experts, 1/2/4/8 concurrent streams"),
    "flash_next_nvfp4": Workload(
        name="flash_next_nvfp4", index=4, L=48, E=512, k=10, H=2048, I=768, fmt="nvfp4",
        pool_mode="shared", pool_bytes=10.7e9, has_shared=True, bias=False, streams=(1,), steps=1000,
        rho=0.9, note="512 experts top-10 + shared expert, NVFP4, one 10.7 GB pool for all layers"),
    "flash_next_prefill": Workload(
        name="flash_next_prefill", index=5, L=48, E=512, k=10, H=2048, I=768, fmt="nvfp4",
        pool_mode="shared", pool_bytes=10.7e9, has_shared=True, bias=True, streams=(1, 4, 16, 32),
        steps=256, rho=0.9, prompt_T=2451,
        note="2451-token prompt through each layer, then decode batches 1/4/16/32"),
}


def scaled(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (smaller test cases)."""
    d = dict(w.__dict__)
    d.update(kw)
    return Workload(**d)
