// route.cu -- the routing kernels of one layer call: router logits, top-k and
// the cache plan (decode), the prefill top-k and read-only plan, the routing
// entry point that allocates nothing, and their launch helpers. The device
// routines they share with the fused decode kernel are in route_dev.cuh.
#include <string.h>

#include <mutex>

#include "../../include/moe_cache.h"
#include "route_dev.cuh"

namespace moe {

// Fused decode routing: all CTAs compute logits; the last CTA to finish
// prefetches the pool's state, ranks every token and runs the plan.
template <int NT>
__global__ void __launch_bounds__(kRouteThreads, 1) k_route(const __grid_constant__ CacheDev c, const __grid_constant__ Scratch s,
                                                         const __grid_constant__ RouteArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    griddep_wait();
    griddep_launch();
    {
        // the pairs' activation maxima start from zero for the expert kernels
        // that follow (the previous call's readers have completed)
        const int P = a.T * c.k + (c.has_shared ? a.T : 0);
        const int nthr = blockDim.x * gridDim.x * gridDim.y;
        for (int i = (blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x; i < P; i += nthr)
            s.act_amax[i] = 0u;
    }
    router_logits_tile<NT>(c, a, smem, s.logits, s.bounds, s.tok_shift);
    if (a.prefill) return;
    __threadfence();
    __syncthreads();
    __shared__ int is_last;
    __shared__ int rerank;
    __shared__ unsigned long long clk;
    if (threadIdx.x == 0) {
        unsigned total = gridDim.x * gridDim.y;
        is_last = atomicAdd(s.route_done, 1u) == total - 1;
        rerank = 0;
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    const int E = c.E, T = a.T, n_ids = T * c.k;
    const int U = min(n_ids, E) + 1;
    const int P = n_ids + (c.has_shared ? T : 0);
    const int pool = c.pool_mode ? 0 : a.layer;
    PlanSmem m = plan_layout(smem, E, c.K, n_ids, U, P);
    const int warp = threadIdx.x >> 5;
    const int nwt = min(kRouteWarps, T);
    const TopkSmem tw = topk_layout(smem + m.bytes + (size_t)warp * topk_bytes_per_warp(E), E);
    if (nwt < kRouteWarps) {
        // the ranking warps start at once; the others stage the pool's state
        if (warp >= nwt) plan_prefetch(c, a, m, pool, threadIdx.x - nwt * 32, blockDim.x - nwt * 32, &clk);
        else
            for (int t = warp; t < T; t += nwt) topk_dispatch(c, s, a, t, tw, &rerank, s.ids, s.wts);
    } else {
        plan_prefetch(c, a, m, pool, threadIdx.x, blockDim.x, &clk);
        for (int t = warp; t < T; t += nwt) topk_dispatch(c, s, a, t, tw, &rerank, s.ids, s.wts);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        *s.route_done = 0;
        s.plan->reranked = rerank;
        if (rerank) c.stats[15] += 1;
    }
    plan_decode(c, s, a, m, clk, s.ids, s.units, true);
}

// Prefill logits: the prompt's tokens in tiles of kRoutePrefillTokens, the
// CTA's kRouteWarps router rows staged in shared memory beside them (not held
// in registers as the decode routing holds them), so two CTAs share an SM.
// The same per-lane sums, butterfly and bounds as k_route's, so the same
// logits; the token prescales come from the CTAs of the first expert column.
constexpr int kRoutePrefillTokens = 16;

__global__ void __launch_bounds__(kRouteThreads, 2) k_route_prefill(const __grid_constant__ CacheDev c,
                                                                   const __grid_constant__ Scratch s,
                                                                   const __grid_constant__ RouteArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    griddep_wait();
    const int H = c.H, E = c.E, NT = kRoutePrefillTokens;
    {
        // the pairs' activation maxima start from zero for the expert kernels
        const int P = a.T * c.k + (c.has_shared ? a.T : 0);
        const int nthr = blockDim.x * gridDim.x * gridDim.y;
        for (int i = (blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x; i < P; i += nthr)
            s.act_amax[i] = 0u;
    }
    const int t0 = blockIdx.y * NT, nt = min(NT, a.T - t0);
    const int e0 = blockIdx.x * kRouteWarps, ne = min(kRouteWarps, E - e0);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);          // [NT][H]
    uint16_t* wr = xs + (size_t)NT * H;                         // [kRouteWarps][H]
    const int vpr = H / 8;
    for (int i = threadIdx.x; i < nt * vpr; i += blockDim.x)
        reinterpret_cast<uint4*>(xs)[i] = reinterpret_cast<const uint4*>(a.x + (size_t)t0 * H)[i];
    for (int i = threadIdx.x; i < ne * vpr; i += blockDim.x)
        reinterpret_cast<uint4*>(wr)[i] = __ldg(reinterpret_cast<const uint4*>(a.w + (size_t)e0 * H) + i);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (blockIdx.x == 0)
        for (int tt = warp; tt < nt; tt += kRouteWarps) {
            const unsigned m = token_absmax_warp(xs + (size_t)tt * H, H, lane);
            if (lane == 0) s.tok_shift[t0 + tt] = token_shift(m);
        }
    if (warp >= ne) return;
    router_logits_warp_smem<kRoutePrefillTokens>(c, a, xs, t0, nt, e0 + warp, wr + (size_t)warp * H, s.logits,
                                                 s.bounds);
}

// Prefill: one warp per token.
__global__ void __launch_bounds__(kRouteThreads) k_topk(const __grid_constant__ CacheDev c, const __grid_constant__ Scratch s,
                                                       const __grid_constant__ RouteArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    griddep_wait();
    const int warp = threadIdx.x >> 5, E = c.E;
    const int t = blockIdx.x * kRouteWarps + warp;
    __shared__ int rerank;
    if (threadIdx.x == 0) rerank = 0;
    __syncthreads();
    const TopkSmem tw = topk_layout(smem + (size_t)warp * topk_bytes_per_warp(E), E);
    if (t < a.T) topk_dispatch(c, s, a, t, tw, &rerank, s.ids, s.wts);
    __syncthreads();
    if (threadIdx.x == 0 && rerank) atomicAdd(c.stats + 15, 1ull);
}

// Prefill plan: read-only lookup. Units: resident experts ascending, then
// staged experts ascending (so groups of `group` are contiguous ranges).
__global__ void __launch_bounds__(1024) k_plan_prefill(CacheDev c, Scratch s, RouteArgs a, int group) {
    extern __shared__ __align__(16) uint8_t smem[];
    griddep_wait();
    const int E = c.E, k = c.k, T = a.T, layer = a.layer;
    const int n_ids = T * k;
    const int P = n_ids + (c.has_shared ? T : 0);
    const int tid = threadIdx.x, nthr = blockDim.x;
    int* used = reinterpret_cast<int*>(smem);  // [E]
    int* unit_of = used + E;                   // [E]
    int* cnt = unit_of + E;                    // [E+2]
    int* cur = cnt + E + 2;                    // [E+2]
    __shared__ int nh_s, nu_s;
    const int* slot_map = c.slot_map + (size_t)layer * E;
    const int pool = c.pool_mode ? 0 : layer;
    for (int e = tid; e < E; e += nthr) used[e] = 0;
    __syncthreads();
    for (int i = tid; i < n_ids; i += nthr) used[s.ids[i]] = 1;
    __syncthreads();
    if (tid == 0) {
        int u = 0;
        for (int e = 0; e < E; ++e)
            if (used[e] && slot_map[e] >= 0) unit_of[e] = u++;
        int nh = u;
        int mi = 0;
        for (int e = 0; e < E; ++e)
            if (used[e] && slot_map[e] < 0) {
                unit_of[e] = u++;
                int half = (mi / group) & 1;
                s.copy_expert[mi] = e;
                s.copy_slot[mi] = -1;
                s.copy_src[mi] = (uint64_t)(c.store + ((size_t)layer * E + e) * c.slot_stride);
                s.copy_dst[mi] = (uint64_t)(c.arena + ((size_t)half * group + (mi % group)) * c.slot_stride);
                mi++;
            }
        nh_s = nh;
        nu_s = u;
    }
    __syncthreads();
    const int nu = nu_s, nh = nh_s;
    const int n_units = nu + (c.has_shared ? 1 : 0);
    for (int u = tid; u <= n_units; u += nthr) cnt[u] = 0;
    __syncthreads();
    for (int i = tid; i < P; i += nthr) {
        int u = i < n_ids ? unit_of[s.ids[i]] : nu;
        s.pair_unit[i] = u;
        atomicAdd(&cnt[u], 1);
    }
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int u = 0; u < n_units; ++u) {
            cur[u] = acc;
            acc += cnt[u];
        }
        cur[n_units] = acc;
    }
    __syncthreads();
    for (int e = tid; e < E; e += nthr) {
        if (!used[e]) continue;
        const int u = unit_of[e];
        const bool hit = slot_map[e] >= 0;
        UnitDesc d;
        d.pstart = cur[u];
        d.np = cnt[u];
        d.expert = e;
        d.slot = hit ? slot_map[e] : -1;
        d.hit = hit;
        d.src = hit ? (uint64_t)(c.pool + ((size_t)pool * c.K + slot_map[e]) * c.slot_stride) : s.copy_dst[u - nh];
        d.dst = 0;
        for (int j = 0; j < 3; ++j) d.g[j] = c.gtable[((size_t)layer * E + e) * 3 + j];
        s.units[u] = d;
    }
    if (tid == 0 && c.has_shared) {
        UnitDesc d;
        d.pstart = cur[nu];
        d.np = cnt[nu];
        d.expert = -1;
        d.slot = -1;
        d.hit = 1;
        d.src = (uint64_t)(c.shared_w + (size_t)layer * c.slot_stride);
        d.dst = 0;
        for (int j = 0; j < 3; ++j) d.g[j] = c.gtable[((size_t)c.L * E + layer) * 3 + j];
        s.units[nu] = d;
    }
    __syncthreads();
    for (int i = tid; i < P; i += nthr) {
        int u = s.pair_unit[i];
        s.unit_pairs[atomicAdd(&cur[u], 1)] = i;
    }
    __syncthreads();
    for (int u = tid; u < n_units; u += nthr) {
        const int st = s.units[u].pstart, n = s.units[u].np;
        for (int j = 0; j < 8; ++j) s.units[u].pair8[j] = j < n ? s.unit_pairs[st + j] : -1;
    }
    if (!c.pagein)
        for (int i = tid; i < n_ids; i += nthr) {
            int e = s.ids[i];
            s.slot_of[i] = slot_map[e];
            s.hit_of[i] = slot_map[e] >= 0;
        }
    __syncthreads();
    if (tid == 0) {
        Plan* pl = s.plan;
        pl->n_uniq = nu;
        pl->n_hit = nh;
        pl->n_fill = nu - nh;
        pl->n_units = n_units;
        pl->status = 0;
        if (c.pagein) return;  // k_pagein commits the transaction, the stats and the trace
        unsigned long long* st = c.stats + a.bucket * 5;
        st[0] += 1;
        st[1] += (unsigned long long)nh;
        st[2] += (unsigned long long)(nu - nh);
        st[3] += (unsigned long long)(nu - nh) * c.slot_bytes;
        if (c.trace) write_trace(c, s, layer, T, n_ids, nh, nu - nh, nu);
    }
}

// ---------------------------------------------------------------------------
// Page-in prefill: "Running an MoE Model Larger Than Your VRAM: SGLang Paged
// Experts, ..." (dev.to), "Why do short prompts get slower first tokens?": a
// prefill pages in every expert it routes to that is not resident, once. The
// cache transaction of decode over all of the call's distinct experts, with
// no capacity rule: the hits are touched in first-occurrence order, then each
// miss, in ascending expert order, takes the least recently used slot and
// becomes the most recently used. With the last-use clock that is: the list
// at the start of the misses is L0 = the untouched slots by ascending stamp,
// then the hits in touch order, and miss j takes slot L0[j mod K] (from the
// K-th miss on, a slot the same call filled or read; only the last miss
// placed in a slot stays). One CTA, after k_plan_prefill (whose units are the
// hits ascending, then the misses ascending). The records still cross the
// host link once, into the staging arena; k_pagein_copy moves those that stay
// resident from the arena into their slots after the GEMMs of their group.
// ---------------------------------------------------------------------------
constexpr int kPageinThreads = 1024;

__host__ __device__ inline size_t pagein_sort_len(int K) {
    size_t n = 1;
    while (n < (size_t)K) n <<= 1;
    return n;
}

// keys [N] u64, L0 [K], first / use_slot / is_hit [E], hit-slot bits [K/32 + 1]:
// at most 211 KB (K = 16384, E = 1024)
static size_t pagein_smem(const CacheDev& c) {
    return pagein_sort_len(c.K) * 8 + (size_t)c.K * 4 + (size_t)c.E * 12 + ((size_t)c.K / 32 + 1) * 4;
}

__global__ void __launch_bounds__(kPageinThreads) k_pagein(CacheDev c, Scratch s, RouteArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    griddep_wait();
    const int E = c.E, K = c.K, k = c.k, layer = a.layer;
    const int pool = c.pool_mode ? 0 : layer;
    const int n_ids = a.T * k;
    const int tid = threadIdx.x, nthr = blockDim.x;
    Plan* pl = s.plan;
    const int nu = pl->n_uniq, nh = pl->n_hit, nm = nu - nh;
    const size_t N = pagein_sort_len(K);
    unsigned long long* key = reinterpret_cast<unsigned long long*>(smem);  // [N] sort keys
    int* L0 = reinterpret_cast<int*>(smem + N * 8);                        // [K]
    int* first = L0 + K;                                                    // [E] first occurrence
    int* use_slot = first + E;                                              // [E] slot read from
    int* is_hit = use_slot + E;                                             // [E]
    unsigned* hit_slot = reinterpret_cast<unsigned*>(is_hit + E);           // [K/32 + 1] bit: a hit's slot
    unsigned long long* g_lu = c.last_use + (size_t)pool * K;
    int* g_kof = c.key_of + (size_t)pool * K;
    int* g_smap = c.slot_map + (size_t)layer * E;
    __shared__ unsigned long long clk;
    __shared__ int Kl;  // slots the pool holds (places whose stamp is not ~0)
    if (tid == 0) {
        clk = c.clock[pool];
        Kl = 0;
    }
    for (int e = tid; e < E; e += nthr) {
        first[e] = 0x7fffffff;
        is_hit[e] = 0;
        use_slot[e] = -1;
    }
    for (int i = tid; i <= K / 32; i += nthr) hit_slot[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n_ids; i += nthr) atomicMin(&first[s.ids[i]], i);
    for (int u = tid; u < nh; u += nthr) {
        const UnitDesc& d = s.units[u];
        is_hit[d.expert] = 1;
        use_slot[d.expert] = d.slot;
        atomicOr(&hit_slot[d.slot >> 5], 1u << (d.slot & 31));
    }
    {
        int n = 0;
        for (int i = tid; i < K; i += nthr) n += g_lu[i] != ~0ull;
        atomicAdd(&Kl, n);
    }
    __syncthreads();
    const int KP = Kl;
    // the untouched slots by ascending last-use stamp (stamps < 2^50, slots < 2^14)
    for (size_t i = tid; i < N; i += nthr)
        key[i] = (i < (size_t)K && !((hit_slot[i >> 5] >> (i & 31)) & 1u) && g_lu[i] != ~0ull)
                     ? ((g_lu[i] << 14) | (unsigned long long)i)
                     : ~0ull;
    __syncthreads();
    for (size_t size = 2; size <= N; size <<= 1)
        for (size_t stride = size >> 1; stride > 0; stride >>= 1) {
            for (size_t i = tid; i < N; i += nthr) {
                const size_t j = i ^ stride;
                if (j > i) {
                    const unsigned long long x = key[i], y = key[j];
                    if ((x > y) == ((i & size) == 0)) {
                        key[i] = y;
                        key[j] = x;
                    }
                }
            }
            __syncthreads();
        }
    for (int i = tid; i < KP - nh; i += nthr) L0[i] = (int)(key[i] & 0x3fffull);
    // then the hits in touch order (first occurrence), stamped clk + rank
    for (int u = tid; u < nh; u += nthr) {
        const UnitDesc& d = s.units[u];
        int rank = 0;
        for (int v = 0; v < nh; ++v) rank += first[s.units[v].expert] < first[d.expert];
        L0[KP - nh + rank] = d.slot;
    }
    __syncthreads();
    // misses: miss j (ascending, staged unit nh + j) is read from slot L0[j mod K]
    for (int j = tid; j < nm; j += nthr) {
        const int e = s.units[nh + j].expert;
        const int sl = L0[j % KP];
        use_slot[e] = sl;
        s.copy_slot[j] = sl;
    }
    // evict what the positions that take a miss held before the call
    const int npos = nm < KP ? nm : KP;
    for (int i = tid; i < npos; i += nthr) {
        const int old = g_kof[L0[i]];
        if (old >= 0) c.slot_map[old] = -1;
    }
    __syncthreads();
    // the last miss placed at each position stays; the hits not displaced keep
    // their touch stamps
    for (int i = tid; i < npos; i += nthr) {
        const int jl = i + KP * ((nm - 1 - i) / KP);
        const int e = s.units[nh + jl].expert;
        const int sl = L0[i];
        g_kof[sl] = layer * E + e;
        g_smap[e] = sl;
        g_lu[sl] = clk + nh + jl;
    }
    for (int r = tid; r < nh; r += nthr)
        if (KP - nh + r >= npos) g_lu[L0[KP - nh + r]] = clk + r;
    for (int i = tid; i < n_ids; i += nthr) {
        const int e = s.ids[i];
        s.slot_of[i] = use_slot[e];
        s.hit_of[i] = is_hit[e];
    }
    __syncthreads();
    if (tid == 0) {
        c.clock[pool] = clk + nh + nm;
        pl->pool_slots = KP;
        unsigned long long* st = c.stats + a.bucket * 5;
        st[0] += 1;
        st[1] += (unsigned long long)nh;
        st[2] += (unsigned long long)nm;
        st[3] += (unsigned long long)nm * c.slot_bytes;
        if (c.trace) write_trace(c, s, layer, a.T, n_ids, nh, nm, nu);
    }
}

// Copies the paged-in records of staging group `group` that stay resident
// (miss j stays when no later miss of the call takes its slot: j >= nm - K)
// from the arena into their slots.
constexpr uint64_t kPageinChunk = 32768;
__global__ void __launch_bounds__(256) k_pagein_copy(CacheDev c, Scratch s, int layer, int group, int G) {
    griddep_wait();
    const Plan* pl = s.plan;
    const int nm = pl->n_uniq - pl->n_hit;
    const int keep_from = nm - (nm < pl->pool_slots ? nm : pl->pool_slots);
    const int j0 = max(group * G, keep_from), j1 = min(group * G + G, nm);
    if (j0 >= j1) return;
    const int pool = c.pool_mode ? 0 : layer;
    const uint64_t bytes = c.slot_bytes;
    const int cpr = (int)((bytes + kPageinChunk - 1) / kPageinChunk);
    const long long total = (long long)(j1 - j0) * cpr;
    for (long long w = blockIdx.x; w < total; w += gridDim.x) {
        const int j = j0 + (int)(w / cpr), ch = (int)(w % cpr);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(s.copy_dst[j]) + (size_t)ch * kPageinChunk;
        uint8_t* dst = c.pool + ((size_t)pool * c.K + s.copy_slot[j]) * c.slot_stride + (size_t)ch * kPageinChunk;
        const uint64_t rem = bytes - (uint64_t)ch * kPageinChunk;
        const int nv = (int)((rem < kPageinChunk ? rem : kPageinChunk) / 16);
        for (int v0 = threadIdx.x; v0 < nv; v0 += 256 * 8) {
            uint4 buf[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int v = v0 + i * 256;
                if (v < nv) buf[i] = __ldcg(reinterpret_cast<const uint4*>(src) + v);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int v = v0 + i * 256;
                if (v < nv) reinterpret_cast<uint4*>(dst)[v] = buf[i];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Adaptive per-layer capacity: "Running a 95 GiB MoE Model on a 32 GiB GPU"
// (busyjay.com), "Decode": as decoding progresses, some capacity moves from
// layers with high hit rates to layers with low hit rates, the total kept.
// After every decode call; every adapt_period * L calls the layer with the
// highest hit rate in the window gives adapt_step slots, one at a time, to
// the layer with the lowest (rates compared exactly as h1 (h2 + m2) against
// h2 (h1 + m1); lower layer first on ties; no move on equal rates; bounds
// adapt_kmin .. K places). The moved slot is the giver's least recently used
// (smallest stamp; its expert evicted, its place left empty with stamp ~0)
// and becomes the taker's least recently used: its lowest empty place,
// stamped below every stamp of that pool. One CTA.
// ---------------------------------------------------------------------------
constexpr int kAdaptThreads = 256;

__global__ void __launch_bounds__(kAdaptThreads) k_adapt(CacheDev c) {
    griddep_wait();
    __shared__ int go, dsel, rsel;
    __shared__ unsigned long long wv[kAdaptThreads / 32];
    __shared__ int wi[kAdaptThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = kAdaptThreads / 32;
    if (tid == 0) {
        go = 0;
        const unsigned long long n = *c.adapt_calls + 1;
        *c.adapt_calls = n;
        if (n % ((unsigned long long)c.adapt_period * c.L) == 0) {
            int d = -1, r = -1;
            for (int l = 0; l < c.L; ++l) {
                const unsigned long long h = c.win[2 * l], t = h + c.win[2 * l + 1];
                if (t == 0) continue;
                if (c.pool_K[l] - c.adapt_step >= c.adapt_kmin) {
                    const unsigned long long hd = d < 0 ? 0 : c.win[2 * d], td = d < 0 ? 0 : hd + c.win[2 * d + 1];
                    if (d < 0 || h * td > hd * t) d = l;
                }
                if (c.pool_K[l] + c.adapt_step <= c.K) {
                    const unsigned long long hr = r < 0 ? 0 : c.win[2 * r], tr = r < 0 ? 0 : hr + c.win[2 * r + 1];
                    if (r < 0 || h * tr < hr * t) r = l;
                }
            }
            if (d >= 0 && r >= 0 && d != r) {
                const unsigned long long hd = c.win[2 * d], td = hd + c.win[2 * d + 1];
                const unsigned long long hr = c.win[2 * r], tr = hr + c.win[2 * r + 1];
                if (hd * tr > hr * td) {
                    go = 1;
                    dsel = d;
                    rsel = r;
                }
            }
            for (int l = 0; l < 2 * c.L; ++l) c.win[l] = 0u;
        }
    }
    __syncthreads();
    if (!go) return;
    const int d = dsel, r = rsel, K = c.K;
    unsigned long long* lud = c.last_use + (size_t)d * K;
    unsigned long long* lur = c.last_use + (size_t)r * K;
    for (int mv = 0; mv < c.adapt_step; ++mv) {
        // the giver's least recently used slot (stamps of slots are distinct)
        unsigned long long v = ~0ull;
        int sl = 0x7fffffff;
        for (int i = tid; i < K; i += kAdaptThreads)
            if (lud[i] < v) {
                v = lud[i];
                sl = i;
            }
        // the taker's lowest empty place
        int fr = 0x7fffffff;
        for (int i = tid; i < K; i += kAdaptThreads)
            if (lur[i] == ~0ull) {
                fr = i;
                break;
            }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            const unsigned long long ov = __shfl_xor_sync(0xffffffffu, v, off);
            const int os = __shfl_xor_sync(0xffffffffu, sl, off);
            if (ov < v || (ov == v && os < sl)) {
                v = ov;
                sl = os;
            }
            fr = min(fr, __shfl_xor_sync(0xffffffffu, fr, off));
        }
        if (lane == 0) {
            wv[warp] = v;
            wi[warp] = sl;
        }
        __shared__ int wf[kAdaptThreads / 32];
        if (lane == 0) wf[warp] = fr;
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < nw; ++w) {
                if (wv[w] < wv[0] || (wv[w] == wv[0] && wi[w] < wi[0])) {
                    wv[0] = wv[w];
                    wi[0] = wi[w];
                }
                wf[0] = min(wf[0], wf[w]);
            }
            const int s = wi[0], t = wf[0];
            const int key = c.key_of[(size_t)d * K + s];
            if (key >= 0) c.slot_map[key] = -1;
            c.key_of[(size_t)d * K + s] = -1;
            lud[s] = ~0ull;
            c.pool_K[d] -= 1;
            c.key_of[(size_t)r * K + t] = -1;
            lur[t] = c.floor_stamp[r];
            c.floor_stamp[r] -= 1;
            c.pool_K[r] += 1;
        }
        __syncthreads();
    }
}

void launch_adapt(const CacheDev& c, cudaStream_t st) { k_adapt<<<1, kAdaptThreads, 0, st>>>(c); }

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------
static size_t topk_smem(int E, int warps) { return (size_t)warps * topk_bytes_per_warp(E); }

size_t route_smem_bytes(const CacheDev& c, int T) {
    const int n_ids = T * c.k;
    const int U = min(n_ids, c.E) + 1;
    const int P = n_ids + (c.has_shared ? T : 0);
    size_t x = (size_t)kRouteTokens * c.H * sizeof(uint16_t);
    size_t last = plan_layout(nullptr, c.E, c.K, n_ids, U, P).bytes + topk_smem(c.E, min(kRouteWarps, T));
    return x > last ? x : last;
}

template <int NT>
static void route_nt(const CacheDev& c, const Scratch& s, const RouteArgs& a, cudaStream_t st, bool pdl) {
    dim3 grid((c.E + kRouteWarps - 1) / kRouteWarps, (a.T + NT - 1) / NT);
    size_t sm = a.prefill ? (size_t)NT * c.H * sizeof(uint16_t) : route_smem_bytes(c, a.T);
    static size_t set_route = 0;
    if (sm > set_route) {
        cudaFuncSetAttribute(k_route<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        set_route = sm;
    }
    launch_ex(k_route<NT>, grid, dim3(kRouteThreads), sm, st, pdl, c, s, a);
}

void launch_route(const CacheDev& c, const Scratch& s, const RouteArgs& a, int /*max_units*/, cudaStream_t st,
                  bool pdl) {
    if (a.prefill) {
        const size_t sm = (size_t)(kRoutePrefillTokens + kRouteWarps) * c.H * sizeof(uint16_t);
        static size_t set = 0;
        if (sm > set) {
            cudaFuncSetAttribute(k_route_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            set = sm;
        }
        const dim3 grid((c.E + kRouteWarps - 1) / kRouteWarps, (a.T + kRoutePrefillTokens - 1) / kRoutePrefillTokens);
        launch_ex(k_route_prefill, grid, dim3(kRouteThreads), sm, st, pdl, c, s, a);
        return;
    }
    if (a.T <= 1) route_nt<1>(c, s, a, st, pdl);
    else if (a.T <= 2) route_nt<2>(c, s, a, st, pdl);
    else if (a.T <= 4) route_nt<4>(c, s, a, st, pdl);
    else route_nt<kRouteTokens>(c, s, a, st, pdl);
}

void launch_topk_prefill(const CacheDev& c, const Scratch& s, const RouteArgs& a, cudaStream_t st) {
    size_t sm = topk_smem(c.E, kRouteWarps);
    static size_t set_topk = 0;
    if (sm > set_topk) {
        cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        set_topk = sm;
    }
    k_topk<<<(a.T + kRouteWarps - 1) / kRouteWarps, kRouteThreads, sm, st>>>(c, s, a);
}

void launch_pagein(const CacheDev& c, const Scratch& s, const RouteArgs& a, cudaStream_t st) {
    const size_t sm = pagein_smem(c);
    static size_t set = 0;
    if (sm > set) {
        cudaFuncSetAttribute(k_pagein, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        set = sm;
    }
    k_pagein<<<1, kPageinThreads, sm, st>>>(c, s, a);
}

void launch_pagein_copy(const CacheDev& c, const Scratch& s, int layer, int group, int G, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    k_pagein_copy<<<sms > 0 ? sms : 148, 256, 0, st>>>(c, s, layer, group, G);
}

void launch_plan_prefill(const CacheDev& c, const Scratch& s, const RouteArgs& a, int group, cudaStream_t st) {
    size_t sm = sizeof(int) * (4 * (size_t)c.E + 4);
    static size_t set_plan = 0;
    if (sm > set_plan) {
        cudaFuncSetAttribute(k_plan_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        set_plan = sm;
    }
    k_plan_prefill<<<1, 1024, sm, st>>>(c, s, a, group);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Router + top-k for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc where they route tokens: allocators that
// must not be re-entered from their own callbacks, embedders that budget every
// byte of device memory up front, and latency-critical loops that cannot take
// cudaMalloc's implicit device synchronisation. For them
// moe_route_topk_noalloc computes one layer's routing (logits, top-k,
// weights) without allocating: its scratch (the logit pairs, their bounds
// and a completion counter) lives in the file-scope array below, which every
// GPU that loads the library holds until the process exits. The array is
// shared by every call on a device and keeps the last call's contents; the
// counter is cleared at the start of each call. Calls whose kernels overlap
// on one GPU race on the array.
// ---------------------------------------------------------------------------
namespace moe {

constexpr int kNoAllocMaxTokens = 32;
constexpr int kNoAllocMaxExperts = 512;
constexpr size_t kNoAllocLogitBytes = (size_t)kNoAllocMaxTokens * kNoAllocMaxExperts * sizeof(float2);
constexpr size_t kNoAllocBoundBytes = (size_t)kNoAllocMaxTokens * kNoAllocMaxExperts * sizeof(float);
constexpr size_t kNoAllocScratchBytes = kNoAllocLogitBytes + kNoAllocBoundBytes + 256;

// [logit pairs][bounds][completion counter]
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// All CTAs compute logits; the last one to finish ranks every token.
template <int NT>
__global__ void __launch_bounds__(kRouteThreads, 1) k_route_noalloc(const __grid_constant__ CacheDev c,
                                                                 const __grid_constant__ Scratch s,
                                                                 const __grid_constant__ RouteArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    router_logits_tile<NT>(c, a, smem, s.logits, s.bounds, nullptr);
    __threadfence();
    __syncthreads();
    __shared__ int is_last;
    __shared__ int rerank;
    if (threadIdx.x == 0) {
        is_last = atomicAdd(s.route_done, 1u) == gridDim.x * gridDim.y - 1;
        rerank = 0;
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    const int warp = threadIdx.x >> 5;
    const int nwt = min(kRouteWarps, a.T);
    const TopkSmem tw = topk_layout(smem + (size_t)warp * topk_bytes_per_warp(c.E), c.E);
    if (warp < nwt)
        for (int t = warp; t < a.T; t += nwt) topk_dispatch(c, s, a, t, tw, &rerank, s.ids, s.wts);
}

template <int NT>
static cudaError_t route_noalloc_nt(const CacheDev& c, const Scratch& s, const RouteArgs& a, size_t sm,
                                    cudaStream_t st) {
    dim3 grid((c.E + kRouteWarps - 1) / kRouteWarps, (a.T + NT - 1) / NT);
    cudaError_t e = cudaFuncSetAttribute(k_route_noalloc<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    k_route_noalloc<NT><<<grid, kRouteThreads, sm, st>>>(c, s, a);
    return cudaGetLastError();
}

}  // namespace moe

namespace {

// Device address of g_noalloc_scratch, looked up once per device (the host
// symbol is only a stand-in and must never be handed to a kernel).
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[64] = {nullptr};

cudaError_t noalloc_scratch(int dev, unsigned char** out) {
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, moe::g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_addr[dev] = p;
    }
    *out = static_cast<unsigned char*>(g_noalloc_addr[dev]);
    return cudaSuccess;
}

}  // namespace

extern "C" moe_status_t moe_route_topk_noalloc(const void* hidden, int32_t T, const void* router_w,
                                               const float* router_bias, int32_t num_experts, int32_t hidden_size,
                                               int32_t top_k, int32_t norm_topk, int32_t* ids, float* weights,
                                               void* stream) {
    if (!hidden || !router_w || !ids || !weights) return MOE_ERR_INVALID;
    if (T < 1 || T > moe::kNoAllocMaxTokens || num_experts < 1 || num_experts > moe::kNoAllocMaxExperts ||
        top_k < 1 || top_k > moe::kMaxTopK || top_k > num_experts || hidden_size < 64 || hidden_size % 64 ||
        hidden_size > 4096)
        return MOE_ERR_INVALID;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    unsigned char* base = nullptr;
    if (noalloc_scratch(dev, &base) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    moe::CacheDev c;
    memset(&c, 0, sizeof c);
    c.E = num_experts;
    c.k = top_k;
    c.H = hidden_size;
    c.norm_topk = norm_topk ? 1 : 0;
    moe::Scratch s;
    memset(&s, 0, sizeof s);
    s.logits = reinterpret_cast<float2*>(base);
    s.bounds = reinterpret_cast<float*>(base + moe::kNoAllocLogitBytes);
    s.route_done = reinterpret_cast<unsigned*>(base + moe::kNoAllocLogitBytes + moe::kNoAllocBoundBytes);
    s.ids = ids;
    s.wts = weights;
    moe::RouteArgs a = {};
    a.x = (const uint16_t*)hidden;
    a.w = (const uint16_t*)router_w;
    a.bias = router_bias;
    a.T = T;
    a.layer = 0;
    a.prefill = 0;
    a.bucket = 0;
    if (cudaMemsetAsync(s.route_done, 0, sizeof(unsigned), st) != cudaSuccess) return MOE_ERR_CUDA;
    const size_t xs = (size_t)moe::kRouteTokens * hidden_size * sizeof(uint16_t);
    const size_t tk = (size_t)min(moe::kRouteWarps, (int)T) * moe::topk_bytes_per_warp(num_experts);
    const size_t sm = xs > tk ? xs : tk;
    cudaError_t e;
    if (T <= 1) e = moe::route_noalloc_nt<1>(c, s, a, sm, st);
    else if (T <= 2) e = moe::route_noalloc_nt<2>(c, s, a, sm, st);
    else if (T <= 4) e = moe::route_noalloc_nt<4>(c, s, a, sm, st);
    else e = moe::route_noalloc_nt<moe::kRouteTokens>(c, s, a, sm, st);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
