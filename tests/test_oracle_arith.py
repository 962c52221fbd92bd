"""Pins for the slot and byte arithmetic against the numbers the pages print."""
import os

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _page():
    vals = {}
    for line in open(os.path.join(GOLDEN, "page_arithmetic.txt")):
        if line.strip() and not line.startswith("#"):
            name, value = line.split()[:2]
            vals[name] = float(value)
    return vals


def test_explainer_bus_arithmetic():
    p = _page()
    H, I, L, E, k = 2560, 640, 48, 512, 10
    per_expert = oracle.slot_bytes("q4_0", H, I)
    assert round(3 * H * I / 1e6, 2) == p["explainer_params_per_expert_M"]
    assert round(per_expert / 2 ** 20, 2) == p["explainer_expert_MiB"]
    assert L * E == p["explainer_all_experts"]
    assert round(L * E * per_expert / 2 ** 30, 1) == p["explainer_all_experts_GiB"]
    assert L * k == p["explainer_touched_per_token"]
    per_token = L * k * per_expert
    assert round(per_token / 2 ** 20) == p["explainer_MiB_per_token"]
    assert round(per_token / 31.5e9 * 1e3, 1) == p["explainer_pcie4_ms"]
    assert round(per_token / 63e9 * 1e3, 1) == p["explainer_pcie5_ms"]
    # 4090: 10.7 GiB of slots is 16.9% of the experts; misses at 77% hits
    slots = oracle.slots_for_budget(p["explainer_4090_cache_GiB"] * 2 ** 30, per_expert)
    assert slots == 4155
    assert round(100 * slots / (L * E), 1) == p["explainer_4090_cache_frac_pct"]
    assert round(p["explainer_MiB_per_token"] * (1 - p["explainer_4090_hit_pct"] / 100)) == p["explainer_4090_miss_MiB"]
    assert round(p["explainer_MiB_per_token"] * (1 - p["explainer_5090_hit_pct"] / 100)) == p["explainer_5090_miss_MiB"]
    # the NVMe build's repacked expert blocks have exactly this size
    assert per_expert == p["nvme_block_bytes"]


def test_t4_group_slot_count():
    p = _page()
    L, E = 48, 128
    per_expert = p["t4_experts_GiB"] * 2 ** 30 / (L * E)
    per_group_budget = p["t4_budget_MiB"] * 2 ** 20 / 2  # two 24-layer groups
    slots = oracle.slots_for_budget(per_group_budget, per_expert)
    assert slots == p["t4_group_slots"]
    assert round(100 * slots / (24 * E), 1) == p["t4_group_cover_pct"]


def test_paged_preflight_arithmetic():
    p = _page()
    L, E, k = 48, 128, 8
    assert round(p["paged_int4_expert_MB"] * L) == p["paged_int4_slot_MB"]
    assert round(p["paged_fp8_expert_MB"] * L) == p["paged_fp8_slot_MB"]
    assert 92 // k == p["paged_int4_batch_cap"]
    assert 40 // k == p["paged_fp8_batch_cap"]
    assert 26 // k == p["paged_laptop_batch_cap"]
    assert round(100 * (1 - 92 / E)) == p["paged_int4_random_miss_pct"]
    assert round(100 * (1 - 40 / E)) == p["paged_fp8_random_miss_pct"]
    assert round(100 * (1 - 26 / E)) == p["paged_laptop_random_miss_pct"]


def test_workload_pool_sizes():
    # one shared 10.7 GB pool of NVFP4 experts at H 2048, I 768
    assert oracle.slots_for_budget(10.7e9, oracle.slot_bytes("nvfp4", 2048, 768)) == 4031
    # 92 Q4_0 slots per layer over 48 layers
    assert round(92 * 48 * oracle.slot_bytes("q4_0", 2048, 768) / 1e9, 2) == 11.72
    # the pinned host store that holds every expert of every layer
    assert round(48 * 128 * oracle.slot_bytes("q4_0", 2048, 768) / 1e9, 1) == 16.3
    assert round(48 * 512 * oracle.slot_bytes("nvfp4", 2048, 768) / 1e9, 1) == 65.2
    # budget edge: a pool one byte short of a slot has none
    rb = oracle.slot_bytes("q4_0", 2048, 768)
    assert oracle.slots_for_budget(rb - 1, rb) == 0 and oracle.slots_for_budget(rb, rb) == 1
