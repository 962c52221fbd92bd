// layer.cu -- a whole decode call of one MoE layer in one persistent kernel.
//
// The call is the method of "Your GPU holds 24 GB. This model is 94 GB. It
// still runs." (cloudmash.blog): router logits and top-k ("The model that
// should not fit"), the cache transaction ("Inside llama.cpp PR #29887: slot
// maps, banks, and only the misses cross PCIe"), the expert FFN read through
// the slots ("The bus problem"), the weighted combine plus the shared expert.
//
// One CTA per SM, all resident at once, with two grid-wide barriers:
//
//   1. Each CTA holds the router rows of its experts in registers, issued
//      before the wait on the preceding grid; it stages the tokens and writes
//      its experts' logit pairs and bounds. It also copies the pool's state
//      (stamps, keys, the layer's slot map) into shared memory: every CTA reads
//      the state before the first barrier, and only CTA 0 writes it, after.
//   -- barrier: every logit is written.
//   2. Every CTA ranks every token and runs the plan itself, from the same
//      logits and the same state, so all CTAs derive the same unit
//      descriptors in their own shared memory: no second round trip through
//      global memory. CTA 0 alone commits the state, the fill list, the stats
//      and the trace. Each CTA then asks L2 for the weight bytes it is about
//      to read (bulk L2 prefetches of resident slots), and its two groups of
//      eight warps compute (unit, 16-row tile) items of gate/up + SwiGLU; a
//      missed unit's tiles are read from the mapped host store and written
//      through to the slot, as in the three-kernel path.
//   -- barrier: every activation is written.
//   3. CTA b computes output row tiles b, b + G, ... of the down projection
//      over every unit and combines them with the router weights.
//
// The arithmetic of every step is the three-kernel path's (same per-warp
// logit sums, same chunk split and warp order in gate/up, the same row-tile
// down projection), so the two paths give bitwise identical results.
//
// Barrier waits are bounded: a wait that outlasts kBarrierTimeoutNs sets an
// error bit the host reports as MOE_ERR_TIMEOUT, and the kernel returns.
#include "expert_dev.cuh"
#include "route_dev.cuh"

namespace moe {

constexpr int kLThreads = 512;
constexpr int kLWarps = kLThreads / 32;
constexpr int kLayerMaxTokens = 8;    // tokens per call (a unit has at most 8 pairs: one n-tile)
constexpr int kLayerMaxPairs = 48;    // T * k (+ T for the shared expert)
constexpr int kLayerRankWarps = 4;    // warps that rank tokens (each needs a TopkSmem)
constexpr unsigned long long kBarrierTimeoutNs = 200ull * 1000 * 1000;
constexpr unsigned kBarrierMaxPolls = 1u << 24;
constexpr size_t kLayerSmemLimit = 224 * 1024;  // dynamic; the static variables take the rest

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~(size_t)15; }

// Shared-memory layout of one call, computed the same way on host and device.
struct LayerLayout {
    size_t sd, ids, wts, xg;     // persistent: descriptors, picks, weights, f16 tokens [T+1][H+8]
    size_t un;                   // start of the phase union
    size_t xs, wr, plan, topk;   // phase 1-2: bf16 tokens [T][H], router rows, the plan, ranking warps
    size_t red;                  // phase 2: gate/up partial tiles [2 groups][8 warps][2][128]
    size_t ah, al, ps;           // phase 3: activations hi/lo, down partials
    size_t total;
};

__host__ __device__ inline LayerLayout layer_layout(int E, int K, int k, int H, int I, int T, int has_shared,
                                                    int rows) {
    LayerLayout L;
    const int n_ids = T * k, U = (n_ids < E ? n_ids : E) + 1, P = n_ids + (has_shared ? T : 0);
    size_t o = 0;
    L.sd = o; o = align16(o + (size_t)U * sizeof(UnitDesc));
    L.ids = o; o = align16(o + (size_t)n_ids * 4);
    L.wts = o; o = align16(o + (size_t)n_ids * 4);
    L.xg = o; o = align16(o + (size_t)(T + 1) * (H + 8) * 2);
    L.un = o;
    // phases 1-2: tokens, plan, ranking
    size_t p = o;
    L.xs = p; p = align16(p + (size_t)T * H * 2);
    L.wr = p; p = align16(p + (size_t)rows * H * 2);
    L.plan = p; p = align16(p + plan_layout(nullptr, E, K, n_ids, U, P).bytes);
    L.topk = p; p = align16(p + (size_t)(T < kLayerRankWarps ? T : kLayerRankWarps) * topk_bytes_per_warp(E));
    size_t end = p;
    // gate/up
    L.red = o;
    p = align16(o + (size_t)2 * 8 * 2 * 128 * 4);
    if (p > end) end = p;
    // down
    const size_t ld = (size_t)I + 8;
    L.ah = o;
    L.al = align16(L.ah + (size_t)(P + 1) * ld * 2);
    L.ps = align16(L.al + (size_t)(P + 1) * ld * 2);
    p = L.ps + down_rows_work_bytes(I, P) - 2 * (size_t)(P + 1) * ld * 2;
    p = align16(p);
    if (p > end) end = p;
    L.total = end;
    return L;
}

// Grid-wide barrier of a grid whose CTAs are all resident. Each CTA adds to
// one counter; CTA 0 adds 2^31 - (G - 1) and the others 1, so the top bit
// flips exactly when the last CTA arrives and the counter needs no reset
// between barriers or calls. Thread 0 of each CTA knows the bit before the
// barrier (`phase`, read once per call), so its arrival is a fire-and-forget
// release add and the wait polls for the flip. Returns false (and sets err)
// if the wait gave up.
__device__ __forceinline__ bool grid_barrier(unsigned* ctr, unsigned* err, unsigned& phase) {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned inc = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1) : 1u;
        asm volatile("red.release.gpu.global.add.u32 [%0], %1;\n" ::"l"(ctr), "r"(inc) : "memory");
        const unsigned long long t0 = globaltimer_ns();
        int good = 1;
        for (unsigned it = 0;; ++it) {
            unsigned cur;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(cur) : "l"(ctr) : "memory");
            if ((cur & 0x80000000u) != phase) break;
            // bounded by time, and by a count in case the timer stalls
            if (globaltimer_ns() - t0 > kBarrierTimeoutNs || it > kBarrierMaxPolls) {
                atomicOr(err, 1u);
                good = 0;
                break;
            }
        }
        phase ^= 0x80000000u;
        ok = good;
    }
    __syncthreads();
    return ok != 0;
}

// Asynchronous global -> shared copies of 4, 8 or 16 bytes (completed by
// cp_async_wait).
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem_dst, const void* gmem_src) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(d), "l"(gmem_src) : "memory");
}

// Asks L2 for [p, p + bytes) of device memory (16-byte aligned start and
// size); the copy runs in the background.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

// The byte range of row tile rt of a slot matrix (R rows, C cols): the codes
// of its chunks, then the scales they use (rounded out to 16 bytes; both stay
// inside the matrix's 16-byte padded extent). Returns the number of ranges.
template <int FMT>
__device__ __forceinline__ int tile_ranges(int R, int C, int rt, uint64_t (&off)[2], uint32_t (&len)[2]) {
    const int KC = C / 64;
    if constexpr (FMT == FMT_Q4_0 || FMT == FMT_NVFP4) {
        off[0] = (uint64_t)rt * KC * 512;
        len[0] = (uint32_t)KC * 512;
        off[1] = (uint64_t)R * C / 2 + (uint64_t)rt * KC * 64;
        len[1] = (uint32_t)KC * 64;
        return 2;
    } else if constexpr (FMT == FMT_FP8_B128) {
        off[0] = (uint64_t)rt * KC * 1024;
        len[0] = (uint32_t)KC * 1024;
        const int nct = (C + 127) / 128;
        const uint64_t s0 = (uint64_t)R * C + (uint64_t)((rt * 16) / 128) * nct * 4;
        const uint64_t s1 = s0 + (uint64_t)nct * 4;
        off[1] = s0 & ~15ull;
        len[1] = (uint32_t)(((s1 + 15) & ~15ull) - off[1]);
        return 2;
    } else {
        off[0] = (uint64_t)rt * KC * 2048;
        len[0] = (uint32_t)KC * 2048;
        return 1;
    }
}

// 16-byte asynchronous copy global -> shared (completed by cp_async_wait).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_all;\n" ::: "memory");
}

// B fragments of the four k-steps of chunk kc, each lane reading its own
// token row (row: this lane's row of the f16 token tile, lane & 7 its column).
__device__ __forceinline__ void load_b_row(const uint16_t* row, int kc, int lane, uint32_t (&b)[4][2]) {
    const uint16_t* p = row + kc * 64 + (lane >> 3) * 8;
    ldmatrix_x4(b[0][0], b[0][1], b[1][0], b[1][1], p);
    ldmatrix_x4(b[2][0], b[2][1], b[3][0], b[3][1], p + 32);
}

__device__ __forceinline__ void group_sync(int group) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(group + 1), "r"(256) : "memory");
}


template <int FMT>
__global__ void __launch_bounds__(kLThreads, 1) k_layer(CacheDev c, Scratch s, RouteArgs a, float* __restrict__ out) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ unsigned long long clk;
    __shared__ int rerank;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const int E = c.E, H = c.H, I = c.I, k = c.k, T = a.T;
    const int n_ids = T * k;
    const int U = min(n_ids, E) + 1;
    const int P = n_ids + (c.has_shared ? T : 0);
    const int pool = c.pool_mode ? 0 : a.layer;
    const int rows = (E + G - 1) / G;
    const LayerLayout L = layer_layout(E, c.K, k, H, I, T, c.has_shared, rows);
    UnitDesc* sd = reinterpret_cast<UnitDesc*>(smem + L.sd);
    int* sids = reinterpret_cast<int*>(smem + L.ids);
    float* swts = reinterpret_cast<float*>(smem + L.wts);
    uint16_t* xg = reinterpret_cast<uint16_t*>(smem + L.xg);
    const int ldx = H + 8;

    // ---- 1. logits ---------------------------------------------------------
    // warp j of CTA b owns expert b + j G; its router row does not depend on
    // the preceding grid, so its copy to shared memory starts before the wait
    // (each lane copies, and later reads, its own 16-byte vectors)
    const int e_mine = b + G * warp;
    uint16_t* wr = reinterpret_cast<uint16_t*>(smem + L.wr) + (size_t)warp * H;
    if (e_mine < E)
        for (int i = 0; i < H / 256; ++i)
            cp_async16(wr + lane * 8 + i * 256, a.w + (size_t)e_mine * H + lane * 8 + i * 256);
    griddep_wait();
    griddep_launch();
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L.xs);
    const PlanSmem m = plan_layout(smem + L.plan, E, c.K, n_ids, U, P);
    unsigned phase = 0;
    {
        // one round of asynchronous copies: the tokens and the pool's state
        // (stamps, keys, the layer's slot map, NVFP4 global scales), read by
        // every CTA before the first barrier (only CTA 0 writes them, after)
        const unsigned long long* lu = c.last_use + (size_t)pool * c.K;
        const int* kof = c.key_of + (size_t)pool * c.K;
        const int* smap = c.slot_map + (size_t)a.layer * E;
        for (int i = tid; i < T * (H / 8); i += kLThreads) cp_async16(xs + (size_t)i * 8, a.x + (size_t)i * 8);
        for (int i = tid; i < c.K; i += kLThreads) {
            cp_async8(m.lu + i, lu + i);
            cp_async4(m.kof + i, kof + i);
        }
        for (int i = tid; i < E; i += kLThreads) {
            cp_async4(m.smap + i, smap + i);
            m.first[i] = 0x7fffffff;
        }
        if (c.fmt == FMT_NVFP4) {
            for (int i = tid; i < E * 3; i += kLThreads) cp_async4(m.gl + i, c.gtable + (size_t)a.layer * E * 3 + i);
            if (tid < 3) cp_async4(m.gl + E * 3 + tid, c.gtable + ((size_t)c.L * E + a.layer) * 3 + tid);
        }
        for (int i = tid; i <= E / 32; i += kLThreads) m.missbits[i] = 0u;
        if (tid == 0) {
            clk = c.clock[pool];
            rerank = 0;
            unsigned cur;
            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];\n" : "=r"(cur) : "l"(s.grid_bar) : "memory");
            phase = cur & 0x80000000u;
        }
        cp_async_wait();
        __syncthreads();
        // f16 copy of the tokens for the expert B operand (converted as the
        // gate/up kernel does); row T is zero
        for (int i = tid; i < T * (H / 8); i += kLThreads) {
            const int t = i / (H / 8), v = i - t * (H / 8);
            const uint4 val = *reinterpret_cast<const uint4*>(xs + (size_t)i * 8);
            uint32_t w4[4] = {val.x, val.y, val.z, val.w};
            if constexpr (FMT != FMT_BF16) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float lo = __uint_as_float(w4[j] << 16);
                    const float hi = __uint_as_float(w4[j] & 0xffff0000u);
                    w4[j] = h2_as_u32(__floats2half2_rn(lo, hi));
                }
            }
            *reinterpret_cast<uint4*>(xg + (size_t)t * ldx + v * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        for (int i = tid; i < ldx / 2; i += kLThreads) reinterpret_cast<uint32_t*>(xg + (size_t)T * ldx)[i] = 0u;
    }
    if (e_mine < E) {
        uint4 wv[kRouterMaxVec];
#pragma unroll
        for (int i = 0; i < kRouterMaxVec; ++i)
            if (i < H / 256) wv[i] = *reinterpret_cast<const uint4*>(wr + lane * 8 + i * 256);
        for (int t = 0; t < T; ++t)
            router_logits_warp<1>(c, a, xs + (size_t)t * H, t, 1, e_mine, wv, s.logits, s.bounds);
    }
    if (!grid_barrier(s.grid_bar, s.err, phase)) return;

    // ---- 2. top-k and plan in every CTA, then gate/up ---------------------
    {
        const int nrw = min(T, kLayerRankWarps);
        if (warp < nrw) {
            const TopkSmem tw = topk_layout(smem + L.topk + (size_t)warp * topk_bytes_per_warp(E), E);
            for (int t = warp; t < T; t += nrw) topk_dispatch(c, s, a, t, tw, &rerank, sids, swts);
        }
    }
    __syncthreads();
    const bool commit = b == 0;
    if (commit) {
        for (int i = tid; i < n_ids; i += kLThreads) {
            s.ids[i] = sids[i];
            s.wts[i] = swts[i];
        }
        if (tid == 0) {
            s.plan->reranked = rerank;
            if (rerank) c.stats[15] += 1;
        }
    }
    plan_small(c, s, a, m, clk, sids, sd, commit);
    const int n_units = m.scal[0] + (c.has_shared ? 1 : 0);
    __syncthreads();  // the gate/up scratch below overlaps the plan's shared memory
    const int RT = I / 16, KC = H / 64;
    const int n_items = n_units * RT;
    const uint64_t mgu = matrix_stride(FMT, I, H);
    // L2 prefetch of the resident bytes this CTA reads: its gate/up items,
    // then its down row tiles of every unit
    {
        const int n_mine = n_items > b ? (n_items - b + G - 1) / G : 0;
        for (int q = tid; q < n_mine * 2; q += kLThreads) {
            const int it = b + G * (q >> 1), u = it / RT, rt = it - u * RT;
            const UnitDesc& d = sd[u];
            if (d.dst) continue;  // a miss: read from the host store
            const uint8_t* M = reinterpret_cast<const uint8_t*>(d.src) + (q & 1) * mgu;
            uint64_t off[2];
            uint32_t len[2];
            const int nr = tile_ranges<FMT>(I, H, rt, off, len);
            for (int r = 0; r < nr; ++r) prefetch_l2(M + off[r], len[r]);
        }
        const int RTD = H / 16;
        const int n_dt = RTD > b ? (RTD - b + G - 1) / G : 0;
        for (int q = tid; q < n_dt * n_units; q += kLThreads) {
            const int u = q % n_units, rt = b + G * (q / n_units);
            const UnitDesc& d = sd[u];
            if (d.dst) continue;
            const uint8_t* M = reinterpret_cast<const uint8_t*>(d.src) + 2 * mgu;
            uint64_t off[2];
            uint32_t len[2];
            const int nr = tile_ranges<FMT>(H, I, rt, off, len);
            for (int r = 0; r < nr; ++r) prefetch_l2(M + off[r], len[r]);
        }
    }
    // gate/up + SwiGLU: group g (warps 8g .. 8g+7) takes items b + G j for
    // j = g, g + 2, ...; the K split over the group's warps, the chunk batches
    // and the warp-ordered sum are the gate/up kernel's
    {
        const int grp = warp >> 3, gw = warp & 7, gtid = tid & 255;
        float* red = reinterpret_cast<float*>(smem + L.red) + (size_t)grp * 8 * 2 * 128;
        const int cpw = (KC + 7) / 8;
        // chunks a warp keeps in flight: fewer than the gate/up kernel's, to
        // stay within 128 registers; the L2 prefetch above hides the rest
        constexpr int CIF = FMT == FMT_BF16 ? 1 : 2;
        for (int j = grp; b + G * j < n_items; j += 2) {
            const int it = b + G * j, u = it / RT, rt = it - u * RT;
            const UnitDesc d = sd[u];
            const uint8_t* Wg = reinterpret_cast<const uint8_t*>(d.src);
            const uint8_t* Wu = Wg + mgu;
            uint8_t* Dg = d.dst ? reinterpret_cast<uint8_t*>(d.dst) : nullptr;
            uint8_t* Du = Dg ? Dg + mgu : nullptr;
            if (Dg && gtid == 0) atomicMin(s.copy_t0, globaltimer_ns());
            if (Dg && rt == 0) {
                copy_matrix_tail<FMT>(Wg, Dg, I, H, gtid, 256);
                copy_matrix_tail<FMT>(Wu, Du, I, H, gtid, 256);
            }
            const int np = d.np;
            // this lane's token row of the B tile (zero row past the unit's pairs)
            const int col = lane & 7;
            const int tok = col < np ? pair_token(pair_at(s, d, col), T, k) : T;
            const uint16_t* brow = xg + (size_t)tok * ldx;
            float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
            for (int c0 = 0; c0 < cpw; c0 += CIF) {
                Chunk<FMT> cg[CIF], cu[CIF];
#pragma unroll
                for (int i = 0; i < CIF; ++i) {
                    const int kc = gw * cpw + c0 + i;
                    if (c0 + i < cpw && kc < KC) {
                        load_chunk<FMT>(Wg, Dg, I, H, rt, kc, lane, cg[i]);
                        load_chunk<FMT>(Wu, Du, I, H, rt, kc, lane, cu[i]);
                    }
                }
#pragma unroll
                for (int i = 0; i < kMaxChunksInFlight; ++i) {
                    const int kc = gw * cpw + c0 + i;
                    if (c0 + i < cpw && kc < KC) {
                        uint32_t bb[1][4][2];
                        load_b_row(brow, kc, lane, bb[0]);
                        mma_chunk<FMT, 1>(cg[i], bb, ag);
                        mma_chunk<FMT, 1>(cu[i], bb, au);
                    }
                }
            }
            const int g = lane >> 2, q = lane & 3;
            float* rg = red + (size_t)(gw * 2) * 128;
            float* ru = rg + 128;
            rg[g * 8 + 2 * q] = ag[0];
            rg[g * 8 + 2 * q + 1] = ag[1];
            rg[(g + 8) * 8 + 2 * q] = ag[2];
            rg[(g + 8) * 8 + 2 * q + 1] = ag[3];
            ru[g * 8 + 2 * q] = au[0];
            ru[g * 8 + 2 * q + 1] = au[1];
            ru[(g + 8) * 8 + 2 * q] = au[2];
            ru[(g + 8) * 8 + 2 * q + 1] = au[3];
            group_sync(grp);
            if (gtid < 128) {
                const int row = gtid >> 3, cc = gtid & 7;
                float gs = 0.f, us = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    gs += red[(size_t)(w * 2) * 128 + gtid];
                    us += red[(size_t)(w * 2 + 1) * 128 + gtid];
                }
                if (cc < np) {
                    const int pair = pair_at(s, d, cc);
                    s.act[(size_t)pair * I + rt * 16 + row] = silu_f(gs * d.g[0]) * (us * d.g[1]);
                }
            }
            if (Dg) {
                // this item's share of the missed record's down matrix
                const uint64_t mdn = matrix_stride(FMT, H, I);
                const uint64_t nvec = mdn / 16, per = (nvec + RT - 1) / RT;
                const uint64_t v0 = (uint64_t)rt * per, v1 = v0 + per < nvec ? v0 + per : nvec;
                const uint8_t* src = Wg + 2 * mgu;
                uint8_t* dst = Dg + 2 * mgu;
                constexpr int kBatch = 4;
                for (uint64_t v = v0 + gtid; v < v1; v += 256ull * kBatch) {
                    uint4 buf[kBatch];
#pragma unroll
                    for (int i = 0; i < kBatch; ++i) {
                        const uint64_t vi = v + (uint64_t)i * 256;
                        if (vi < v1) buf[i] = ldg_stream(src + vi * 16);
                    }
#pragma unroll
                    for (int i = 0; i < kBatch; ++i) {
                        const uint64_t vi = v + (uint64_t)i * 256;
                        if (vi < v1) stg_stream(dst + vi * 16, buf[i]);
                    }
                }
                if (gtid == 0) atomicMax(s.copy_t1, globaltimer_ns());
            }
            group_sync(grp);
        }
    }
    if (!grid_barrier(s.grid_bar, s.err, phase)) return;

    // ---- 3. down projection + combine by row tiles -------------------------
    if (commit && tid == 0) {
        // every miss of the call has been streamed: book the time
        const unsigned long long t1 = atomicAdd(s.copy_t1, 0ull);
        if (t1) {
            const unsigned long long t0 = atomicAdd(s.copy_t0, 0ull);
            c.stats[a.bucket * 5 + 4] += t1 - t0;
            *s.copy_t0 = ~0ull;
            *s.copy_t1 = 0ull;
        }
    }
    const int RTD = H / 16;
    if (b < RTD) {
        uint16_t* ah = reinterpret_cast<uint16_t*>(smem + L.ah);
        uint16_t* al = reinterpret_cast<uint16_t*>(smem + L.al);
        float* ps = reinterpret_cast<float*>(smem + L.ps);
        down_stage_act<FMT>(s, P, I, ah, al);
        __syncthreads();
        for (int rt = b; rt < RTD; rt += G) down_rows_tile<FMT>(c, s, sd, n_units, T, rt, ah, al, ps, swts, out);
    }
}

// ---------------------------------------------------------------------------
// Launch
// ---------------------------------------------------------------------------
static int g_layer_ctas[64];

static int layer_ctas() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!g_layer_ctas[dev]) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_layer_ctas[dev] = sms;
    }
    return g_layer_ctas[dev];
}

size_t layer_smem_bytes(const CacheDev& c, int T) {
    if (T < 1 || T > kLayerMaxTokens) return 0;
    const int P = T * c.k + (c.has_shared ? T : 0);
    const int G = layer_ctas();
    // every expert needs a warp of some CTA
    if (P > kLayerMaxPairs || G <= 0 || (c.E + G - 1) / G > kLWarps) return 0;
    const size_t b = layer_layout(c.E, c.K, c.k, c.H, c.I, T, c.has_shared, (c.E + G - 1) / G).total;
    return b <= kLayerSmemLimit ? b : 0;
}

template <int FMT>
static bool layer_launch(const CacheDev& c, const Scratch& s, const RouteArgs& a, float* out, size_t sm,
                         cudaStream_t st, bool pdl) {
    static size_t set = 0;
    if (sm > set) {
        if (cudaFuncSetAttribute(k_layer<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess)
            return false;
        set = sm;
    }
    // one CTA per SM, all resident: the grid barriers rely on it
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_layer<FMT>, kLThreads, sm) != cudaSuccess ||
        per_sm < 1)
        return false;
    return launch_ex(k_layer<FMT>, dim3(layer_ctas()), dim3(kLThreads), sm, st, pdl, c, s, a, out) == cudaSuccess;
}

bool launch_layer(const CacheDev& c, const Scratch& s, const RouteArgs& a, float* out, int bucket, cudaStream_t st,
                  bool pdl) {
    (void)bucket;
    const size_t sm = layer_smem_bytes(c, a.T);
    if (!sm || !c.fused_upload) return false;
    switch (c.fmt) {
    case FMT_BF16: return layer_launch<FMT_BF16>(c, s, a, out, sm, st, pdl);
    case FMT_Q4_0: return layer_launch<FMT_Q4_0>(c, s, a, out, sm, st, pdl);
    case FMT_FP8_B128: return layer_launch<FMT_FP8_B128>(c, s, a, out, sm, st, pdl);
    case FMT_NVFP4: return layer_launch<FMT_NVFP4>(c, s, a, out, sm, st, pdl);
    }
    return false;
}

}  // namespace moe
