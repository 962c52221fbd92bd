// api.cu -- the C ABI (include/moe_cache.h): handle lifetime, expert loading,
// the per-layer forward (kernel orchestration on the caller's stream), stats,
// trace and state readback.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <string>
#include <thread>
#include <vector>

#include "../../include/moe_cache.h"
#include "common.cuh"
#include "decode_policy.h"

struct moe_cache {
    moe_config_t cfg;
    moe::CacheDev dev;
    moe::Scratch scr;
    int maxT = 0, maxU = 0, maxP = 0, G = 32;
    uint64_t record_bytes = 0, slot_bytes = 0, slot_stride = 0;
    uint64_t pool_bytes_dev = 0, store_bytes = 0, scratch_bytes = 0;
    uint8_t* store_host = nullptr;
    std::vector<uint8_t> loaded;  // [L*E]
    std::vector<uint8_t> shared_loaded;
    size_t n_loaded = 0, n_shared_loaded = 0;
    std::vector<void*> dev_allocs;
    std::string err;
    // MOE_UPLOAD_MEMCPY: pinned readback of the fill list
    int* host_fill = nullptr;  // [2 + 2*maxU]
    uint64_t memcpy_upload_ns[3] = {0, 0, 0};
    int trace_cap = 0, trace_stride = 0;
    std::vector<float> gtable_host;
    // per-stage event timing
    bool prof_on = false;
    bool fused_ok = true;  // the one-kernel decode path launched (or was not tried yet)
    uint64_t fused_calls = 0, split_calls = 0;
    int last_layer = -1;    // layer of the previous layer call on this handle (-1: none since reset)
    std::vector<cudaEvent_t> ev_pool;
    size_t ev_used = 0;
    // prefill staging: a side stream copies group g + 1 into one half of the
    // arena while the tensor-core GEMMs of group g read the other half
    cudaStream_t stage_stream = nullptr;
    cudaEvent_t ev_plan = nullptr, ev_copy[2] = {nullptr, nullptr}, ev_gemm[2] = {nullptr, nullptr};
    struct Span { int stage, a, b; };
    std::vector<Span> spans;
    // speculative next-layer routing: the registered routers, the side stream,
    // its events per layer parity and the layer whose prefetch is in flight
    std::vector<const void*> spec_w;
    std::vector<const float*> spec_b;
    cudaStream_t spec_stream = nullptr;
    cudaEvent_t ev_route[2] = {nullptr, nullptr}, ev_spec_plan[2] = {nullptr, nullptr},
                ev_spec_copy[2] = {nullptr, nullptr};
    float* spec_z = nullptr;
    unsigned* spec_done = nullptr;
    int spec_pending = -1;
};

namespace {

thread_local std::string g_create_error;

moe_status_t fail(moe_cache_t* h, moe_status_t st, const std::string& msg) {
    if (h) h->err = msg;
    else g_create_error = msg;
    return st;
}

moe_status_t cuda_fail(moe_cache_t* h, cudaError_t e, const char* what) {
    return fail(h, MOE_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define CK(h, call)                                        \
    do {                                                   \
        cudaError_t e_ = (call);                           \
        if (e_ != cudaSuccess) return cuda_fail(h, e_, #call); \
    } while (0)

template <typename T>
cudaError_t dalloc(moe_cache_t* h, T** p, size_t n) {
    void* q = nullptr;
    cudaError_t e = cudaMalloc(&q, n * sizeof(T) > 0 ? n * sizeof(T) : 16);
    if (e == cudaSuccess) h->dev_allocs.push_back(q);
    *p = reinterpret_cast<T*>(q);
    return e;
}

int prof_event(moe_cache_t* h, cudaStream_t st) {
    if (h->ev_used == h->ev_pool.size()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return -1;
        h->ev_pool.push_back(e);
    }
    cudaEventRecord(h->ev_pool[h->ev_used], st);
    return (int)h->ev_used++;
}

// Brackets one launch with events when profiling is on.
template <typename F>
void timed(moe_cache_t* h, int stage, cudaStream_t st, F&& launch) {
    if (!h->prof_on) { launch(); return; }
    int a = prof_event(h, st);
    launch();
    int b = prof_event(h, st);
    if (a >= 0 && b >= 0) h->spans.push_back({stage, a, b});
}

void free_all(moe_cache_t* h) {
    for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
    h->ev_pool.clear();
    for (cudaEvent_t* e : {&h->ev_plan, &h->ev_copy[0], &h->ev_copy[1], &h->ev_gemm[0], &h->ev_gemm[1]}) {
        if (*e) cudaEventDestroy(*e);
        *e = nullptr;
    }
    if (h->stage_stream) cudaStreamDestroy(h->stage_stream);
    h->stage_stream = nullptr;
    for (int i = 0; i < 2; ++i)
        for (cudaEvent_t* e : {&h->ev_route[i], &h->ev_spec_plan[i], &h->ev_spec_copy[i]}) {
            if (*e) cudaEventDestroy(*e);
            *e = nullptr;
        }
    if (h->spec_stream) cudaStreamDestroy(h->spec_stream);
    h->spec_stream = nullptr;
    for (void* p : h->dev_allocs) cudaFree(p);
    h->dev_allocs.clear();
    if (h->store_host) cudaFreeHost(h->store_host);
    h->store_host = nullptr;
    if (h->host_fill) cudaFreeHost(h->host_fill);
    h->host_fill = nullptr;
}

// Initial cache state: all slots empty, stamps 0..K-1 (slot 0 least recent).
moe_status_t init_tables(moe_cache_t* h) {
    const moe::CacheDev& d = h->dev;
    std::vector<int> sm((size_t)d.L * d.E, -1), ko((size_t)d.n_pools * d.K, -1);
    std::vector<unsigned long long> lu((size_t)d.n_pools * d.K), clk(d.n_pools, (unsigned long long)d.K);
    for (int p = 0; p < d.n_pools; ++p)
        for (int s = 0; s < d.K; ++s) lu[(size_t)p * d.K + s] = (unsigned long long)s;
    if (d.adapt_period) {
        // places 0..K0-1 hold the slots at the start; the stamps start at 2^32
        // so slots that arrive later can be stamped below all of them
        const unsigned long long base = 1ull << 32;
        const int K0 = h->cfg.slots_per_layer;
        for (int p = 0; p < d.n_pools; ++p) {
            for (int s = 0; s < d.K; ++s) lu[(size_t)p * d.K + s] = s < K0 ? base + s : ~0ull;
            clk[p] = base + K0;
        }
        std::vector<int> pk(d.n_pools, K0);
        std::vector<unsigned long long> fl(d.n_pools, base - 1);
        CK(h, cudaMemcpy(d.pool_K, pk.data(), pk.size() * sizeof(int), cudaMemcpyHostToDevice));
        CK(h, cudaMemcpy(d.floor_stamp, fl.data(), fl.size() * sizeof(unsigned long long), cudaMemcpyHostToDevice));
        CK(h, cudaMemset(d.win, 0, 2 * (size_t)d.L * sizeof(unsigned)));
        CK(h, cudaMemset(d.adapt_calls, 0, sizeof(unsigned long long)));
    }
    CK(h, cudaMemcpy(d.slot_map, sm.data(), sm.size() * sizeof(int), cudaMemcpyHostToDevice));
    CK(h, cudaMemcpy(d.key_of, ko.data(), ko.size() * sizeof(int), cudaMemcpyHostToDevice));
    CK(h, cudaMemcpy(d.last_use, lu.data(), lu.size() * sizeof(unsigned long long), cudaMemcpyHostToDevice));
    CK(h, cudaMemcpy(d.clock, clk.data(), clk.size() * sizeof(unsigned long long), cudaMemcpyHostToDevice));
    CK(h, cudaMemset(d.stats, 0, 18 * sizeof(unsigned long long)));
    if (d.bank_n) {
        CK(h, cudaMemset(d.bank_n, 0, 2 * sizeof(int)));
        CK(h, cudaMemset(d.bank_key, 0xff, 2 * (size_t)d.bank_half * sizeof(int)));
    }
    h->spec_pending = -1;
    CK(h, cudaMemset(d.uses, 0, (size_t)d.L * d.E * sizeof(unsigned)));
    if (h->scr.grid_bar) CK(h, cudaMemset(h->scr.grid_bar, 0, sizeof(unsigned)));
    if (h->scr.err) CK(h, cudaMemset(h->scr.err, 0, sizeof(unsigned)));
    if (h->scr.logit_ctr) CK(h, cudaMemset(h->scr.logit_ctr, 0, 2 * sizeof(unsigned)));
    if (h->scr.pass_ctr) CK(h, cudaMemset(h->scr.pass_ctr, 0, 2 * sizeof(unsigned)));
    if (d.trace_count) CK(h, cudaMemset(d.trace_count, 0, sizeof(unsigned long long)));
    memset(h->memcpy_upload_ns, 0, sizeof(h->memcpy_upload_ns));
    return MOE_OK;
}

bool valid_fmt(int f) { return f >= MOE_FMT_BF16 && f <= MOE_FMT_NVFP4; }

}  // namespace

extern "C" {

void moe_config_default(moe_config_t* cfg) {
    if (!cfg) return;
    memset(cfg, 0, sizeof(*cfg));
    cfg->format = MOE_FMT_BF16;
    cfg->pool_mode = MOE_POOL_PER_LAYER;
    cfg->upload_mode = MOE_UPLOAD_PULL;
    cfg->norm_topk = 1;
    cfg->max_cache_tokens = 32;
    cfg->prefill_group = 32;
    cfg->max_tokens = 32;
    cfg->device = 0;
    cfg->split_decode = MOE_DECODE_AUTO;
    cfg->multi_wave = 0;
    cfg->eviction = MOE_EVICT_LRU;
    cfg->speculate = 0;
    cfg->prefill_mode = MOE_PREFILL_READ_ONLY;
    cfg->adapt_period = 0;
    cfg->adapt_step = 0;
    cfg->adapt_min_slots = 0;
    cfg->adapt_max_slots = 0;
}

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_last_error(const moe_cache_t* h) {
    if (h) return h->err.c_str();
    return g_create_error.c_str();
}

moe_status_t moe_cache_create(const moe_config_t* cfg, const void* const* expert_host,
                              const void* const* shared_host, moe_cache_t** out) {
    if (!out) return fail(nullptr, MOE_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (!cfg) return fail(nullptr, MOE_ERR_INVALID, "cfg is NULL");
    const moe_config_t c = *cfg;
    if (c.num_layers < 1 || c.num_experts < 1 || c.num_experts > moe::kMaxExperts)
        return fail(nullptr, MOE_ERR_INVALID, "num_layers must be >= 1 and num_experts in 1..1024");
    if (c.top_k < 1 || c.top_k > moe::kMaxTopK || c.top_k > c.num_experts)
        return fail(nullptr, MOE_ERR_INVALID, "top_k must be in 1..min(16, num_experts)");
    if (c.hidden < 64 || c.hidden % 64 || c.inter < 64 || c.inter % 64)
        return fail(nullptr, MOE_ERR_INVALID, "hidden and inter must be positive multiples of 64");
    if (c.hidden > 4096 || c.inter > 4096) return fail(nullptr, MOE_ERR_INVALID, "hidden and inter must be <= 4096");
    if (!valid_fmt(c.format)) return fail(nullptr, MOE_ERR_INVALID, "unknown format");
    if (c.pool_mode != MOE_POOL_PER_LAYER && c.pool_mode != MOE_POOL_SHARED)
        return fail(nullptr, MOE_ERR_INVALID, "unknown pool_mode");
    if (c.upload_mode != MOE_UPLOAD_PULL && c.upload_mode != MOE_UPLOAD_MEMCPY)
        return fail(nullptr, MOE_ERR_INVALID, "unknown upload_mode");
    if (c.split_decode < MOE_DECODE_AUTO || c.split_decode > MOE_DECODE_ONE_KERNEL)
        return fail(nullptr, MOE_ERR_INVALID, "unknown decode mode (split_decode)");
    if (c.multi_wave != 0 && c.multi_wave != 1) return fail(nullptr, MOE_ERR_INVALID, "multi_wave must be 0 or 1");
    if (c.eviction != MOE_EVICT_LRU && c.eviction != MOE_EVICT_LFU)
        return fail(nullptr, MOE_ERR_INVALID, "unknown eviction policy");
    if (c.speculate != 0 && c.speculate != 1) return fail(nullptr, MOE_ERR_INVALID, "speculate must be 0 or 1");
    if (c.speculate && c.upload_mode != MOE_UPLOAD_PULL)
        return fail(nullptr, MOE_ERR_INVALID, "speculation needs MOE_UPLOAD_PULL");
    if (c.prefill_mode != MOE_PREFILL_READ_ONLY && c.prefill_mode != MOE_PREFILL_PAGE_IN)
        return fail(nullptr, MOE_ERR_INVALID, "unknown prefill_mode");
    if (c.prefill_mode == MOE_PREFILL_PAGE_IN && c.eviction != MOE_EVICT_LRU)
        return fail(nullptr, MOE_ERR_INVALID, "the page-in prefill needs LRU eviction");
    moe_config_t cc = c;  // with the adaptive capacity's defaults filled in
    if (cc.adapt_period < 0) return fail(nullptr, MOE_ERR_INVALID, "adapt_period must be >= 0");
    if (cc.adapt_period > 0) {
        if (cc.pool_mode != MOE_POOL_PER_LAYER)
            return fail(nullptr, MOE_ERR_INVALID, "adaptive capacity needs per-layer pools");
        if (cc.adapt_step == 0) cc.adapt_step = 1;
        if (cc.adapt_min_slots == 0) cc.adapt_min_slots = std::max(cc.top_k, cc.slots_per_layer / 2);
        if (cc.adapt_max_slots == 0) cc.adapt_max_slots = 2 * cc.slots_per_layer - cc.adapt_min_slots;
        if (cc.adapt_step < 1 || cc.adapt_min_slots < cc.top_k || cc.adapt_min_slots > cc.slots_per_layer ||
            cc.adapt_max_slots < cc.slots_per_layer || cc.adapt_max_slots > 16384)
            return fail(nullptr, MOE_ERR_INVALID,
                        "adaptive capacity needs top_k <= adapt_min_slots <= slots_per_layer <= adapt_max_slots "
                        "<= 16384 and adapt_step >= 1");
    }
    if (c.max_cache_tokens < 1 || c.max_cache_tokens > moe::kDecodeMaxTokens)
        return fail(nullptr, MOE_ERR_INVALID, "max_cache_tokens must be in 1..32");
    if (c.max_tokens < 1) return fail(nullptr, MOE_ERR_INVALID, "max_tokens must be >= 1");
    if (c.prefill_group < 1 || c.prefill_group > 1024) return fail(nullptr, MOE_ERR_INVALID, "prefill_group in 1..1024");

    moe_cache_t* h = new moe_cache();
    h->cfg = cc;
    moe::CacheDev& d = h->dev;
    d.L = c.num_layers; d.E = c.num_experts; d.k = c.top_k; d.H = c.hidden; d.I = c.inter;
    d.fmt = c.format; d.has_shared = c.has_shared ? 1 : 0; d.norm_topk = c.norm_topk ? 1 : 0;
    d.pool_mode = c.pool_mode;
    d.fused_upload = c.upload_mode == MOE_UPLOAD_PULL ? 1 : 0;
    const uint64_t cgu = moe::matrix_bytes(d.fmt, d.I, d.H), cdn = moe::matrix_bytes(d.fmt, d.H, d.I);
    h->record_bytes = 2 * cgu + cdn + (d.fmt == moe::FMT_NVFP4 ? 12 : 0);
    h->slot_bytes = 2 * moe::matrix_stride(d.fmt, d.I, d.H) + moe::matrix_stride(d.fmt, d.H, d.I);
    h->slot_stride = (h->slot_bytes + 255) & ~255ull;
    d.slot_bytes = h->slot_bytes;
    d.slot_stride = h->slot_stride;
    if (c.pool_mode == MOE_POOL_PER_LAYER) {
        d.n_pools = d.L;
        d.K = cc.adapt_period ? cc.adapt_max_slots : c.slots_per_layer;
        d.adapt_period = cc.adapt_period;
        d.adapt_step = cc.adapt_step;
        d.adapt_kmin = cc.adapt_min_slots;
    } else {
        d.n_pools = 1;
        double k = c.pool_bytes > 0 ? floor(c.pool_bytes / (double)h->slot_bytes) : 0.0;
        d.K = k > 1e9 ? 1000000000 : (int)k;
    }
    if ((c.pool_mode == MOE_POOL_PER_LAYER ? c.slots_per_layer : d.K) < d.k) {
        char msg[160];
        snprintf(msg, sizeof msg, "pool has %d slots, fewer than top_k = %d", d.K, d.k);
        delete h;
        return fail(nullptr, MOE_ERR_CAPACITY, msg);
    }
    if (d.K > 16384) {
        delete h;
        return fail(nullptr, MOE_ERR_INVALID, "at most 16384 slots per pool");
    }
    h->maxT = c.max_tokens;
    h->G = c.prefill_group;
    h->maxU = std::min(h->maxT * d.k, d.E) + 1;
    h->maxP = h->maxT * d.k + h->maxT;

    cudaError_t e = cudaSetDevice(c.device);
    if (e != cudaSuccess) { delete h; return cuda_fail(nullptr, e, "cudaSetDevice"); }

    auto bail = [&](moe_status_t st, const std::string& m) {
        free_all(h);
        delete h;
        return fail(nullptr, st, m);
    };
#define DA(ptr, n)                                                                \
    do {                                                                          \
        cudaError_t e2 = dalloc(h, &(ptr), (n));                                  \
        if (e2 != cudaSuccess) return bail(MOE_ERR_OOM, std::string("device allocation of ") + #ptr + " failed"); \
    } while (0)

    // pinned store: every expert of every layer, in slot layout
    h->store_bytes = (uint64_t)d.L * d.E * h->slot_stride;
    e = cudaHostAlloc((void**)&h->store_host, h->store_bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) { h->store_host = nullptr; return bail(MOE_ERR_OOM, "pinned host store allocation failed"); }
    void* store_dev = nullptr;
    e = cudaHostGetDevicePointer(&store_dev, h->store_host, 0);
    if (e != cudaSuccess) return bail(MOE_ERR_CUDA, "cudaHostGetDevicePointer failed");
    d.store = (const uint8_t*)store_dev;
    h->loaded.assign((size_t)d.L * d.E, 0);
    h->shared_loaded.assign(d.L, 0);

    uint8_t *pool = nullptr, *sharedw = nullptr, *arena = nullptr;
    h->pool_bytes_dev = (uint64_t)d.n_pools * d.K * h->slot_stride;
    DA(pool, h->pool_bytes_dev);
    d.pool = pool;
    if (d.has_shared) { DA(sharedw, (size_t)d.L * h->slot_stride); d.shared_w = sharedw; }
    if (h->maxT > c.max_cache_tokens) { DA(arena, (size_t)2 * h->G * h->slot_stride); d.arena = arena; }
    float* gt = nullptr;
    DA(gt, ((size_t)d.L * d.E + d.L) * 3);
    d.gtable = gt;
    h->gtable_host.assign(((size_t)d.L * d.E + d.L) * 3, 1.0f);
    if (cudaMemcpy(gt, h->gtable_host.data(), h->gtable_host.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
        return bail(MOE_ERR_CUDA, "gtable upload failed");
    DA(d.slot_map, (size_t)d.L * d.E);
    DA(d.key_of, (size_t)d.n_pools * d.K);
    DA(d.last_use, (size_t)d.n_pools * d.K);
    DA(d.clock, (size_t)d.n_pools);
    DA(d.uses, (size_t)d.L * d.E);
    d.lfu = c.eviction == MOE_EVICT_LFU ? 1 : 0;
    d.pagein = c.prefill_mode == MOE_PREFILL_PAGE_IN ? 1 : 0;
    DA(d.stats, 18);
    if (d.adapt_period) {
        DA(d.pool_K, (size_t)d.n_pools);
        DA(d.win, 2 * (size_t)d.L);
        DA(d.adapt_calls, 1);
        DA(d.floor_stamp, (size_t)d.n_pools);
    }
    h->spec_w.assign(d.L, nullptr);
    h->spec_b.assign(d.L, nullptr);
    if (c.speculate) {
        // the prefetch bank: two halves (layer parity) of top_k x kSpecMaxTokens slots
        d.bank_half = d.k * moe::kSpecMaxTokens;
        uint8_t* bank = nullptr;
        DA(bank, 2 * (size_t)d.bank_half * h->slot_stride);
        d.bank = bank;
        DA(d.bank_key, 2 * (size_t)d.bank_half);
        DA(d.bank_n, 2);
        DA(h->spec_z, (size_t)moe::kSpecMaxTokens * d.E);
        DA(h->spec_done, 1);
        if (cudaMemset(h->spec_done, 0, 4) != cudaSuccess) return bail(MOE_ERR_CUDA, "scratch initialisation failed");
        if (cudaStreamCreateWithFlags(&h->spec_stream, cudaStreamNonBlocking) != cudaSuccess)
            return bail(MOE_ERR_CUDA, "speculation stream creation failed");
        for (int i = 0; i < 2; ++i)
            for (cudaEvent_t* ev : {&h->ev_route[i], &h->ev_spec_plan[i], &h->ev_spec_copy[i]})
                if (cudaEventCreateWithFlags(ev, cudaEventDisableTiming) != cudaSuccess)
                    return bail(MOE_ERR_CUDA, "speculation event creation failed");
    }
    DA(d.trace_count, 1);
    d.trace = nullptr;
    d.trace_cap = 0;
    h->trace_stride = 6 + 5 * h->maxT * d.k;
    d.trace_stride = h->trace_stride;

    moe::Scratch& s = h->scr;
    const size_t T = h->maxT, U = h->maxU, P = h->maxP;
    DA(s.logits, T * d.E);
    DA(s.bounds, T * d.E);
    DA(s.ids, T * d.k);
    DA(s.wts, T * d.k);
    DA(s.slot_of, T * d.k);
    DA(s.hit_of, T * d.k);
    DA(s.units, U);
    DA(s.unit_pairs, P);
    DA(s.pair_unit, P);
    DA(s.copy_src, U);
    DA(s.copy_dst, U);
    DA(s.copy_expert, U);
    DA(s.copy_slot, U);
    DA(s.act, P * d.I);
    DA(s.part, P * d.H);
    DA(s.tok_shift, T);
    DA(s.act_amax, P);
    DA(s.pass_ctr, 2);
    DA(s.plan, 1);
    DA(s.route_done, 1);
    DA(s.tile_done, (size_t)d.H / 16);
    DA(s.copy_done, 1);
    DA(s.copy_t0, 1);
    DA(s.copy_t1, 1);
    DA(s.tiles_done, 1);
    DA(s.grid_bar, 1);
    DA(s.err, 1);
    DA(s.logit_ctr, 2);
    if (h->maxT > c.max_cache_tokens) {
        DA(s.gemm_items, moe::gemm_max_items(P, U));
        DA(s.gemm_count, 1);
        if (cudaStreamCreateWithFlags(&h->stage_stream, cudaStreamNonBlocking) != cudaSuccess)
            return bail(MOE_ERR_CUDA, "staging stream creation failed");
        for (cudaEvent_t* ev : {&h->ev_plan, &h->ev_copy[0], &h->ev_copy[1], &h->ev_gemm[0], &h->ev_gemm[1]})
            if (cudaEventCreateWithFlags(ev, cudaEventDisableTiming) != cudaSuccess)
                return bail(MOE_ERR_CUDA, "staging event creation failed");
    }
#undef DA
    h->scratch_bytes = T * d.E * 16 + T * d.k * 16 + U * (sizeof(moe::UnitDesc) + 32) + P * 8 + P * (d.I + d.H) * 4;
    if (cudaMemset(s.route_done, 0, 4) != cudaSuccess || cudaMemset(s.tile_done, 0, (d.H / 16) * 4) != cudaSuccess ||
        cudaMemset(s.copy_done, 0, 4) != cudaSuccess || cudaMemset(s.copy_t0, 0xff, 8) != cudaSuccess ||
        cudaMemset(s.copy_t1, 0, 8) != cudaSuccess || cudaMemset(s.plan, 0, sizeof(moe::Plan)) != cudaSuccess ||
        cudaMemset(s.tiles_done, 0, 4) != cudaSuccess || cudaMemset(s.grid_bar, 0, 4) != cudaSuccess ||
        cudaMemset(s.err, 0, 4) != cudaSuccess || cudaMemset(s.logit_ctr, 0, 8) != cudaSuccess ||
        cudaMemset(s.tok_shift, 0, T * sizeof(int)) != cudaSuccess || cudaMemset(s.act_amax, 0, P * 4) != cudaSuccess ||
        cudaMemset(s.pass_ctr, 0, 2 * sizeof(unsigned)) != cudaSuccess)
        return bail(MOE_ERR_CUDA, "scratch initialisation failed");
    if (c.upload_mode == MOE_UPLOAD_MEMCPY) {
        e = cudaHostAlloc((void**)&h->host_fill, sizeof(int) * (2 + 2 * U), cudaHostAllocDefault);
        if (e != cudaSuccess) { h->host_fill = nullptr; return bail(MOE_ERR_OOM, "pinned fill buffer failed"); }
    }
    if (init_tables(h) != MOE_OK) {
        std::string m = h->err;
        return bail(MOE_ERR_CUDA, m);
    }
    if (expert_host) {
        for (int l = 0; l < d.L; ++l) {
            if (!expert_host[l]) continue;
            moe_status_t st = moe_cache_load_experts(h, l, 0, d.E, expert_host[l]);
            if (st != MOE_OK) { std::string m = h->err; return bail(st, m); }
        }
    }
    if (shared_host && d.has_shared) {
        for (int l = 0; l < d.L; ++l) {
            if (!shared_host[l]) continue;
            moe_status_t st = moe_cache_load_shared(h, l, shared_host[l]);
            if (st != MOE_OK) { std::string m = h->err; return bail(st, m); }
        }
    }
    *out = h;
    return MOE_OK;
}

moe_status_t moe_cache_load_experts(moe_cache_t* h, int32_t layer, int32_t first, int32_t count,
                                    const void* records) {
    if (!h) return fail(nullptr, MOE_ERR_INVALID, "handle is NULL");
    const moe::CacheDev& d = h->dev;
    if (!records || layer < 0 || layer >= d.L || first < 0 || count < 0 || first + count > d.E)
        return fail(h, MOE_ERR_INVALID, "bad layer/expert range or NULL records");
    const uint8_t* src = (const uint8_t*)records;
    std::vector<float> g((size_t)count * 3);
    unsigned nth = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
    nth = std::min<unsigned>(nth, (unsigned)std::max(1, count));
    std::atomic<int> next(0);
    auto work = [&]() {
        for (int i = next++; i < count; i = next++) {
            const int e = first + i;
            uint8_t* dst = h->store_host + ((size_t)layer * d.E + e) * h->slot_stride;
            moe::repack_record(d.fmt, d.H, d.I, src + (size_t)i * h->record_bytes, dst, &g[(size_t)i * 3]);
        }
    };
    std::vector<std::thread> th;
    for (unsigned t = 1; t < nth; ++t) th.emplace_back(work);
    work();
    for (auto& t : th) t.join();
    for (int i = 0; i < count; ++i)
        for (int j = 0; j < 3; ++j) h->gtable_host[((size_t)layer * d.E + first + i) * 3 + j] = g[(size_t)i * 3 + j];
    CK(h, cudaMemcpy((float*)d.gtable + ((size_t)layer * d.E + first) * 3, &h->gtable_host[((size_t)layer * d.E + first) * 3],
                     (size_t)count * 3 * sizeof(float), cudaMemcpyHostToDevice));
    for (int i = 0; i < count; ++i) {
        uint8_t& f = h->loaded[(size_t)layer * d.E + first + i];
        if (!f) { f = 1; h->n_loaded++; }
    }
    if (d.bank_n) {
        // records may have changed: nothing prefetched before stays valid
        CK(h, cudaDeviceSynchronize());
        CK(h, cudaMemset(d.bank_n, 0, 2 * sizeof(int)));
        h->spec_pending = -1;
    }
    return MOE_OK;
}

moe_status_t moe_cache_load_shared(moe_cache_t* h, int32_t layer, const void* record) {
    if (!h) return fail(nullptr, MOE_ERR_INVALID, "handle is NULL");
    const moe::CacheDev& d = h->dev;
    if (!d.has_shared) return fail(h, MOE_ERR_INVALID, "the configuration has no shared expert");
    if (!record || layer < 0 || layer >= d.L) return fail(h, MOE_ERR_INVALID, "bad layer or NULL record");
    std::vector<uint8_t> tmp(h->slot_stride, 0);
    float g[3];
    moe::repack_record(d.fmt, d.H, d.I, (const uint8_t*)record, tmp.data(), g);
    CK(h, cudaMemcpy((uint8_t*)d.shared_w + (size_t)layer * h->slot_stride, tmp.data(), h->slot_stride,
                     cudaMemcpyHostToDevice));
    for (int j = 0; j < 3; ++j) h->gtable_host[((size_t)d.L * d.E + layer) * 3 + j] = g[j];
    CK(h, cudaMemcpy((float*)d.gtable + ((size_t)d.L * d.E + layer) * 3, g, sizeof g, cudaMemcpyHostToDevice));
    if (!h->shared_loaded[layer]) { h->shared_loaded[layer] = 1; h->n_shared_loaded++; }
    return MOE_OK;
}

moe_status_t moe_layer_forward(moe_cache_t* h, const void* hidden, int32_t T, const void* router_w,
                               const float* router_bias, int32_t layer_id, float* out, void* stream) {
    if (!h) return fail(nullptr, MOE_ERR_INVALID, "handle is NULL");
    const moe::CacheDev& d = h->dev;
    if (!hidden || !router_w || !out) return fail(h, MOE_ERR_INVALID, "NULL hidden, router_w or out");
    if (layer_id < 0 || layer_id >= d.L) return fail(h, MOE_ERR_INVALID, "layer_id out of range");
    if (T <= 0 || T > h->maxT) return fail(h, MOE_ERR_INVALID, "T must be in 1..max_tokens");
    if (h->n_loaded != (size_t)d.L * d.E || (d.has_shared && h->n_shared_loaded != (size_t)d.L))
        return fail(h, MOE_ERR_STATE, "experts not loaded");
    cudaStream_t st = (cudaStream_t)stream;
    const bool decode = T <= h->cfg.max_cache_tokens;
    // the single-wave rule: a pool whose capacity adapts is held to its minimum
    const int cap = d.adapt_period ? d.adapt_kmin : d.K;
    if (decode && (int64_t)T * d.k > cap) {
        if (!h->cfg.multi_wave)
            return fail(h, MOE_ERR_CAPACITY, "tokens * top_k exceeds the slots of this layer's pool");
        // Several waves, each within the single-wave rule: floor(K / k) tokens
        // per wave (at least one, since create requires K >= k), in token
        // order, each its own cache transaction.
        const int per_wave = cap / d.k;
        for (int t0 = 0; t0 < T; t0 += per_wave) {
            const int tw = std::min(per_wave, T - t0);
            const moe_status_t r = moe_layer_forward(h, (const uint16_t*)hidden + (size_t)t0 * d.H, tw, router_w,
                                                     router_bias, layer_id, out + (size_t)t0 * d.H, stream);
            if (r != MOE_OK) return r;
        }
        return MOE_OK;
    }
    const int bucket = T <= 8 ? 0 : (T <= 32 ? 1 : 2);
    moe::RouteArgs a = {};
    a.x = (const uint16_t*)hidden;
    a.w = (const uint16_t*)router_w;
    a.bias = router_bias;
    a.T = T;
    a.layer = layer_id;
    a.prefill = decode ? 0 : 1;
    a.bucket = bucket;
    // Per-layer pools: this layer's state was last written by its own previous
    // call. When the call just before this one on the handle was another
    // layer's, that write belongs to a grid at least two back in stream order,
    // which has completed by the time this call's kernel can start.
    a.early = (d.pool_mode == 0 && !d.adapt_period && h->last_layer >= 0 && h->last_layer != layer_id) ? 1 : 0;
    h->last_layer = layer_id;
    const int units = std::min(T * d.k, d.E) + d.has_shared;
    // Speculation: the side stream's prefetch for layer spec_pending. Its bank
    // keys are ordered before this call's routing; when it was made for this
    // call, its copies are ordered before this call's expert kernels (below),
    // otherwise before everything of this call.
    bool use_bank = false;
    if (h->spec_pending >= 0) {
        const int half = h->spec_pending & 1;
        CK(h, cudaStreamWaitEvent(st, h->ev_spec_plan[half], 0));
        if (h->spec_pending == layer_id && decode && T <= moe::kSpecMaxTokens) {
            use_bank = true;
        } else {
            CK(h, cudaStreamWaitEvent(st, h->ev_spec_copy[half], 0));
            h->spec_pending = -1;
        }
    }
    a.spec = use_bank ? 1 : 0;
    // programmatic dependent launch between the decode kernels (off while
    // events bracket each launch for profiling)
    const bool pdl = !h->prof_on;
    bool fused = false;
    // the path's rule (and its measured reasons) is in decode_policy.h
    moe::DecodeCall dc;
    dc.mode = h->cfg.split_decode;
    dc.T = T;
    dc.pool_mode = d.pool_mode;
    dc.upload_mode = h->cfg.upload_mode;
    dc.speculate = h->cfg.speculate != 0;
    dc.fused_ok = h->fused_ok;
    dc.fits = decode && moe::layer_smem_bytes(d, T) > 0;
    if (decode && moe::one_kernel_decode(dc)) {
        // the whole call in one persistent kernel
        timed(h, 6, st, [&] { fused = moe::launch_layer(d, h->scr, a, out, bucket, st, pdl); });
        if (!fused) {
            // not launchable here (e.g. one CTA per SM does not fit): clear the
            // launch error and keep to the three-kernel path from now on
            cudaGetLastError();
            h->fused_ok = false;
            if (h->prof_on && !h->spans.empty()) h->spans.pop_back();
        }
    }
    if (decode) ++(fused ? h->fused_calls : h->split_calls);
    if (decode && !fused) {
        // PULL: misses are pulled over the host link by the gate/up kernel,
        // which streams each missed record into its slot while it consumes it
        timed(h, 0, st, [&] { moe::launch_route(d, h->scr, a, units, st, pdl); });
        if (use_bank) {
            // this call's prefetched records must have landed before its expert kernels read them
            CK(h, cudaStreamWaitEvent(st, h->ev_spec_copy[layer_id & 1], 0));
            h->spec_pending = -1;
        }
        if (h->cfg.speculate && T <= moe::kSpecMaxTokens && layer_id + 1 < d.L && h->spec_w[layer_id + 1]) {
            // the next layer's router on this call's tokens, on the side
            // stream after this call's routing (its plan and everything
            // before it), then the predicted non-resident records into the
            // bank half of the next layer, beside this call's expert kernels
            const int nl = layer_id + 1, half = nl & 1;
            CK(h, cudaEventRecord(h->ev_route[half], st));
            CK(h, cudaStreamWaitEvent(h->spec_stream, h->ev_route[half], 0));
            moe::SpecArgs sa;
            sa.x = a.x;
            sa.w = (const uint16_t*)h->spec_w[nl];
            sa.bias = h->spec_b[nl];
            sa.T = T;
            sa.layer = nl;
            sa.half = half;
            sa.z = h->spec_z;
            sa.done = h->spec_done;
            moe::launch_spec_route(d, sa, h->spec_stream);
            CK(h, cudaEventRecord(h->ev_spec_plan[half], h->spec_stream));
            moe::launch_spec_copy(d, half, h->spec_stream);
            CK(h, cudaEventRecord(h->ev_spec_copy[half], h->spec_stream));
            h->spec_pending = nl;
        }
        if (h->cfg.upload_mode == MOE_UPLOAD_MEMCPY) {
            // read the fill list back, then one copy per merged run
            int* hf = h->host_fill;
            CK(h, cudaMemcpyAsync(hf, &h->scr.plan->n_fill, sizeof(int), cudaMemcpyDeviceToHost, st));
            CK(h, cudaStreamSynchronize(st));
            const int nf = hf[0];
            if (nf > 0) {
                CK(h, cudaMemcpyAsync(hf + 2, h->scr.copy_expert, sizeof(int) * nf, cudaMemcpyDeviceToHost, st));
                CK(h, cudaMemcpyAsync(hf + 2 + h->maxU, h->scr.copy_slot, sizeof(int) * nf, cudaMemcpyDeviceToHost, st));
                CK(h, cudaStreamSynchronize(st));
                const int* fe = hf + 2;
                const int* fs = hf + 2 + h->maxU;
                const int pool = d.pool_mode ? 0 : layer_id;
                auto t0 = std::chrono::steady_clock::now();
                for (int i = 0; i < nf;) {
                    int n = 1;
                    while (i + n < nf && fe[i + n] == fe[i] + n && fs[i + n] == fs[i] + n) ++n;
                    const uint8_t* src = h->store_host + ((size_t)layer_id * d.E + fe[i]) * h->slot_stride;
                    uint8_t* dst = d.pool + ((size_t)pool * d.K + fs[i]) * h->slot_stride;
                    CK(h, cudaMemcpyAsync(dst, src, (size_t)n * h->slot_stride, cudaMemcpyHostToDevice, st));
                    i += n;
                }
                CK(h, cudaStreamSynchronize(st));
                h->memcpy_upload_ns[bucket] += (uint64_t)std::chrono::duration_cast<std::chrono::nanoseconds>(
                                                   std::chrono::steady_clock::now() - t0)
                                                   .count();
            }
        }
        timed(h, 2, st, [&] { moe::launch_gateup(d, h->scr, a.x, T, 0, 0, h->G, units, st, pdl); });
        timed(h, 3, st, [&] {
            if (!moe::launch_down_rows(d, h->scr, out, T, units, bucket, st, pdl))
                moe::launch_down(d, h->scr, out, T, 0, 0, h->G, units, bucket, st, pdl);
        });
    } else if (!decode) {
        timed(h, 0, st, [&] { moe::launch_route(d, h->scr, a, units, st, false); });
        timed(h, 4, st, [&] { moe::launch_topk_prefill(d, h->scr, a, st); });
        timed(h, 5, st, [&] { moe::launch_plan_prefill(d, h->scr, a, h->G, st); });
        if (d.pagein) timed(h, 5, st, [&] { moe::launch_pagein(d, h->scr, a, st); });
        const int groups = (std::min(T * d.k, d.E) + h->G - 1) / h->G;
        if (moe::gemm_supported(d)) {
            // tensor-core grouped GEMMs: resident units and the shared expert in
            // place, then each staging group through the arena; one combine.
            // Group g + 1 is staged over the host link on the side stream into
            // the arena half group g - 1 used, while the GEMMs of group g run:
            // events order each copy after the GEMMs that last read its half
            // and each group's GEMMs after its copy.
            cudaStream_t cs = h->stage_stream;
            CK(h, cudaEventRecord(h->ev_plan, st));
            CK(h, cudaStreamWaitEvent(cs, h->ev_plan, 0));
            timed(h, 2, st, [&] { moe::launch_gemm(d, h->scr, a.x, T, 1, 0, h->G, units, st); });
            for (int g = 0; g < groups; ++g) {
                if (g >= 2) CK(h, cudaStreamWaitEvent(cs, h->ev_gemm[g & 1], 0));
                timed(h, 1, cs, [&] { moe::launch_copy(d, h->scr, g * h->G, h->G, bucket, cs, true); });
                CK(h, cudaEventRecord(h->ev_copy[g & 1], cs));
                CK(h, cudaStreamWaitEvent(st, h->ev_copy[g & 1], 0));
                timed(h, 2, st, [&] { moe::launch_gemm(d, h->scr, a.x, T, 2, g, h->G, h->G, st); });
                // page-in: the group's records that stay resident go to their slots
                // (after the resident units' GEMMs, before the arena half is restaged)
                if (d.pagein) timed(h, 1, st, [&] { moe::launch_pagein_copy(d, h->scr, layer_id, g, h->G, st); });
                CK(h, cudaEventRecord(h->ev_gemm[g & 1], st));
            }
            timed(h, 3, st, [&] { moe::launch_combine(d, h->scr, out, T, st); });
        } else {
            timed(h, 2, st, [&] { moe::launch_gateup(d, h->scr, a.x, T, 1, 0, h->G, units, st, false); });
            timed(h, 3, st, [&] { moe::launch_down(d, h->scr, out, T, 1, 0, h->G, units, bucket, st, false); });
            for (int g = 0; g < groups; ++g) {
                timed(h, 1, st, [&] { moe::launch_copy(d, h->scr, g * h->G, h->G, bucket, st, false); });
                timed(h, 2, st, [&] { moe::launch_gateup(d, h->scr, a.x, T, 2, g, h->G, h->G, st, false); });
                timed(h, 3, st, [&] { moe::launch_down(d, h->scr, out, T, 2, g, h->G, h->G, bucket, st, false); });
                if (d.pagein) timed(h, 1, st, [&] { moe::launch_pagein_copy(d, h->scr, layer_id, g, h->G, st); });
            }
        }
    }
    if (decode && d.adapt_period) moe::launch_adapt(d, st);  // counts the call; moves capacity on its period
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
    return MOE_OK;
}

moe_status_t moe_cache_pool_slots(moe_cache_t* h, int32_t* sizes) {
    if (!h || !sizes) return fail(h, MOE_ERR_INVALID, "NULL argument");
    const moe::CacheDev& d = h->dev;
    CK(h, cudaSetDevice(h->cfg.device));
    CK(h, cudaDeviceSynchronize());
    if (d.pool_K) CK(h, cudaMemcpy(sizes, d.pool_K, sizeof(int) * (size_t)d.n_pools, cudaMemcpyDeviceToHost));
    else
        for (int p = 0; p < d.n_pools; ++p) sizes[p] = d.K;
    return MOE_OK;
}

moe_status_t moe_cache_set_router(moe_cache_t* h, int32_t layer, const void* router_w, const float* router_bias) {
    if (!h) return fail(nullptr, MOE_ERR_INVALID, "handle is NULL");
    if (layer < 0 || layer >= h->dev.L) return fail(h, MOE_ERR_INVALID, "layer out of range");
    h->spec_w[layer] = router_w;
    h->spec_b[layer] = router_w ? router_bias : nullptr;
    return MOE_OK;
}

moe_status_t moe_cache_stats(moe_cache_t* h, moe_stats_t* out) {
    if (!h || !out) return fail(h, MOE_ERR_INVALID, "NULL argument");
    CK(h, cudaSetDevice(h->cfg.device));
    CK(h, cudaDeviceSynchronize());
    unsigned long long st[18];
    CK(h, cudaMemcpy(st, h->dev.stats, sizeof st, cudaMemcpyDeviceToHost));
    memset(out, 0, sizeof(*out));
    for (int b = 0; b < 3; ++b) {
        out->bucket[b].calls = st[b * 5 + 0];
        out->bucket[b].hits = st[b * 5 + 1];
        out->bucket[b].misses = st[b * 5 + 2];
        out->bucket[b].bytes_uploaded = st[b * 5 + 3];
        out->bucket[b].upload_ns = st[b * 5 + 4] + h->memcpy_upload_ns[b];
    }
    out->num_pools = h->dev.n_pools;
    out->slots_per_pool = h->dev.K;
    out->slot_bytes = h->slot_bytes;
    out->record_bytes = h->record_bytes;
    out->topk_fp64_rerank = st[15];
    out->spec_prefetched = st[16];
    out->spec_used = st[17];
    unsigned derr = 0;
    CK(h, cudaMemcpy(&derr, h->scr.err, sizeof derr, cudaMemcpyDeviceToHost));
    if (derr & 1u) return fail(h, MOE_ERR_TIMEOUT, "a grid barrier of the one-kernel decode path timed out");
    if (derr & 2u) return fail(h, MOE_ERR_TIMEOUT, "a weight-slot wait of the one-kernel decode path timed out");
    if (derr & 4u) return fail(h, MOE_ERR_TIMEOUT, "a tensor-core wait of the prefill GEMM timed out");
    return MOE_OK;
}

moe_status_t moe_cache_info(moe_cache_t* h, moe_info_t* out) {
    if (!h || !out) return fail(h, MOE_ERR_INVALID, "NULL argument");
    out->num_pools = h->dev.n_pools;
    out->slots_per_pool = h->dev.K;
    out->slot_bytes = h->slot_bytes;
    out->slot_stride = h->slot_stride;
    out->record_bytes = h->record_bytes;
    out->pool_device_bytes = h->pool_bytes_dev;
    out->store_host_bytes = h->store_bytes;
    out->scratch_device_bytes = h->scratch_bytes;
    out->fused_decode_calls = h->fused_calls;
    out->split_decode_calls = h->split_calls;
    return MOE_OK;
}

moe_status_t moe_cache_trace_enable(moe_cache_t* h, int32_t capacity_calls) {
    if (!h || capacity_calls < 0) return fail(h, MOE_ERR_INVALID, "bad argument");
    CK(h, cudaSetDevice(h->cfg.device));
    CK(h, cudaDeviceSynchronize());
    if (h->dev.trace) {
        cudaFree(h->dev.trace);
        h->dev_allocs.erase(std::remove(h->dev_allocs.begin(), h->dev_allocs.end(), (void*)h->dev.trace),
                            h->dev_allocs.end());
        h->dev.trace = nullptr;
    }
    h->dev.trace_cap = 0;
    h->trace_cap = 0;
    CK(h, cudaMemset(h->dev.trace_count, 0, sizeof(unsigned long long)));
    if (capacity_calls == 0) return MOE_OK;
    int* tr = nullptr;
    if (dalloc(h, &tr, (size_t)capacity_calls * h->trace_stride) != cudaSuccess)
        return fail(h, MOE_ERR_OOM, "trace allocation failed");
    h->dev.trace = tr;
    h->dev.trace_cap = capacity_calls;
    h->trace_cap = capacity_calls;
    return MOE_OK;
}

moe_status_t moe_cache_trace_read(moe_cache_t* h, int32_t* buf, int64_t buf_words, int64_t* n_words,
                                  int32_t* n_records) {
    if (!h || !n_words || !n_records) return fail(h, MOE_ERR_INVALID, "NULL argument");
    *n_words = 0;
    *n_records = 0;
    CK(h, cudaSetDevice(h->cfg.device));
    CK(h, cudaDeviceSynchronize());
    if (!h->dev.trace) return MOE_OK;
    unsigned long long cnt = 0;
    CK(h, cudaMemcpy(&cnt, h->dev.trace_count, sizeof cnt, cudaMemcpyDeviceToHost));
    const unsigned long long have = std::min<unsigned long long>(cnt, (unsigned long long)h->trace_cap);
    std::vector<int> ring((size_t)h->trace_cap * h->trace_stride);
    CK(h, cudaMemcpy(ring.data(), h->dev.trace, ring.size() * sizeof(int), cudaMemcpyDeviceToHost));
    int64_t w = 0;
    for (unsigned long long i = cnt - have; i < cnt; ++i) {
        const int* r = ring.data() + (size_t)(i % h->trace_cap) * h->trace_stride;
        const int64_t len = 6 + 3 * (int64_t)r[2] + 2 * (int64_t)r[4];
        if (buf == nullptr || w + len > buf_words) return fail(h, MOE_ERR_INVALID, "trace buffer too small");
        memcpy(buf + w, r, (size_t)len * sizeof(int));
        w += len;
    }
    *n_words = w;
    *n_records = (int32_t)have;
    CK(h, cudaMemset(h->dev.trace_count, 0, sizeof(unsigned long long)));
    return MOE_OK;
}

moe_status_t moe_cache_get_state(moe_cache_t* h, int32_t* slot_map, int32_t* key_of, int32_t* order) {
    if (!h) return fail(nullptr, MOE_ERR_INVALID, "handle is NULL");
    const moe::CacheDev& d = h->dev;
    CK(h, cudaSetDevice(h->cfg.device));
    CK(h, cudaDeviceSynchronize());
    if (slot_map) CK(h, cudaMemcpy(slot_map, d.slot_map, sizeof(int) * (size_t)d.L * d.E, cudaMemcpyDeviceToHost));
    if (key_of) CK(h, cudaMemcpy(key_of, d.key_of, sizeof(int) * (size_t)d.n_pools * d.K, cudaMemcpyDeviceToHost));
    if (order) {
        std::vector<unsigned long long> lu((size_t)d.n_pools * d.K);
        CK(h, cudaMemcpy(lu.data(), d.last_use, lu.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
        for (int p = 0; p < d.n_pools; ++p) {
            // the places that hold a slot (stamp not ~0), least recent first
            const unsigned long long* v = lu.data() + (size_t)p * d.K;
            std::vector<int> idx;
            for (int s = 0; s < d.K; ++s)
                if (v[s] != ~0ull) idx.push_back(s);
            std::sort(idx.begin(), idx.end(), [&](int a, int b) { return v[a] < v[b]; });
            idx.resize(d.K, -1);
            memcpy(order + (size_t)p * d.K, idx.data(), sizeof(int) * d.K);
        }
    }
    return MOE_OK;
}

moe_status_t moe_cache_read_slot(moe_cache_t* h, int32_t pool, int32_t slot, void* dst, int32_t layer,
                                 int32_t expert, void* store_dst, uint64_t bytes) {
    if (!h) return fail(nullptr, MOE_ERR_INVALID, "handle is NULL");
    const moe::CacheDev& d = h->dev;
    if (pool < 0 || pool >= d.n_pools || slot < 0 || slot >= d.K || bytes > h->slot_stride)
        return fail(h, MOE_ERR_INVALID, "bad pool, slot or size");
    CK(h, cudaSetDevice(h->cfg.device));
    CK(h, cudaDeviceSynchronize());
    if (dst) CK(h, cudaMemcpy(dst, d.pool + ((size_t)pool * d.K + slot) * h->slot_stride, bytes, cudaMemcpyDeviceToHost));
    if (store_dst) {
        if (layer < 0 || layer >= d.L || expert < 0 || expert >= d.E)
            return fail(h, MOE_ERR_INVALID, "bad layer or expert");
        memcpy(store_dst, h->store_host + ((size_t)layer * d.E + expert) * h->slot_stride, bytes);
    }
    return MOE_OK;
}

moe_status_t moe_cache_profile_enable(moe_cache_t* h, int32_t on) {
    if (!h) return fail(nullptr, MOE_ERR_INVALID, "handle is NULL");
    h->prof_on = on != 0;
    return MOE_OK;
}

moe_status_t moe_cache_profile_read(moe_cache_t* h, moe_profile_t* out) {
    if (!h || !out) return fail(h, MOE_ERR_INVALID, "NULL argument");
    memset(out, 0, sizeof(*out));
    CK(h, cudaSetDevice(h->cfg.device));
    CK(h, cudaDeviceSynchronize());
    for (const auto& sp : h->spans) {
        float ms = 0.f;
        CK(h, cudaEventElapsedTime(&ms, h->ev_pool[sp.a], h->ev_pool[sp.b]));
        out->ms[sp.stage] += ms;
        out->launches[sp.stage] += 1;
    }
    h->spans.clear();
    h->ev_used = 0;
    return MOE_OK;
}

moe_status_t moe_cache_reset(moe_cache_t* h) {
    if (!h) return fail(nullptr, MOE_ERR_INVALID, "handle is NULL");
    CK(h, cudaSetDevice(h->cfg.device));
    CK(h, cudaDeviceSynchronize());
    h->last_layer = -1;
    return init_tables(h);
}

moe_status_t moe_cache_destroy(moe_cache_t* h) {
    if (!h) return MOE_OK;
    cudaSetDevice(h->cfg.device);
    cudaDeviceSynchronize();
    free_all(h);
    delete h;
    return MOE_OK;
}

}  // extern "C"
