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
//   1. Each CTA copies the router rows of its experts to shared memory
//      before the wait on the preceding grid; it stages the tokens and writes
//      its experts' logit pairs and bounds. It also copies the pool's state
//      (stamps, keys, the layer's slot map) into shared memory: every CTA reads
//      the state before the first barrier, and only the committing CTA writes
//      it, after.
//   -- barrier: every logit is written.
//   2. Every CTA ranks every token and runs the plan itself, from the same
//      logits and the same state, so all CTAs derive the same unit
//      descriptors in their own shared memory: no second round trip through
//      global memory. One CTA (the last) commits the state, the fill list,
//      the stats and the trace.
//      The CTA then knows every weight byte it will read in this call: the
//      gate/up rows of its (unit, 16-row tile) items and the down rows of its
//      output tiles. It streams the resident ones into a ring of shared-memory
//      slots with bulk copies (the tensor-memory-access engine, completion on
//      one mbarrier per slot, L2 evict-first so streamed weights do not push
//      out the code, the router and the pool state), so HBM sees the whole
//      call's bytes requested at once; each slot is refilled with the next
//      piece as soon as its consumers are done. Two groups of eight warps
//      compute gate/up + SwiGLU from the slots; a missed unit's tiles are read
//      from the mapped host store and written through to the slot, as in the
//      three-kernel path.
//   -- barrier: every activation is written.
//   3. CTA b computes output row tiles b, b + G, ... of the down projection
//      over every unit from the down pieces already in its slots, and
//      combines them with the router weights.
//
// The arithmetic of every step is the three-kernel path's (same per-warp
// logit sums, same chunk split and warp order in gate/up, the same row-tile
// down projection), so the two paths give bitwise identical results.
//
// Waits are bounded: a grid barrier or a slot wait that outlasts its limit
// sets an error bit the host reports as MOE_ERR_TIMEOUT; the kernel waits
// (again bounded) for its own copies in flight before it returns.
#include "decode_policy.h"
#include "expert_dev.cuh"
#include "route_dev.cuh"

namespace moe {

constexpr int kLThreads = 512;
constexpr int kLWarps = kLThreads / 32;
// Warps of a CTA that compute router logits, one expert each: one per
// scheduler, so each logit's instruction stream issues without competing.
constexpr int kLogitWarps = 4;
constexpr int kLayerMaxTokens = 8;    // tokens per call (a unit has at most 8 pairs: one n-tile)
constexpr int kLayerMaxPairs = 48;    // T * k (+ T for the shared expert)
constexpr int kLayerRankWarps = 4;    // warps that rank tokens (each needs a TopkSmem)
constexpr int kMaxSlots = 16;         // ring slots
constexpr unsigned long long kBarrierTimeoutNs = 200ull * 1000 * 1000;
constexpr unsigned kBarrierMaxPolls = 1u << 24;
constexpr unsigned long long kSlotTimeoutNs = 200ull * 1000 * 1000;
constexpr unsigned kSlotMaxPolls = 1u << 26;
constexpr size_t kLayerSmemLimit = 224 * 1024;  // dynamic; the static variables take the rest

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~(size_t)15; }
__host__ __device__ inline size_t align128(size_t v) { return (v + 127) & ~(size_t)127; }

// Upper bound on the bytes of one 16-row tile of a slot matrix with C
// columns: its codes plus its scales (tile_ranges below gives the exact
// ranges; block-FP8's scale range is rounded out to 16 bytes).
__host__ __device__ inline size_t tile_bytes_bound(int fmt, int C) {
    const size_t KC = (size_t)C / 64;
    switch (fmt) {
    case FMT_Q4_0:
    case FMT_NVFP4: return KC * 576;
    case FMT_FP8_B128: return KC * 1024 + align16((size_t)((C + 127) / 128) * 4) + 16;
    default: return KC * 2048;
    }
}

// Shared-memory layout of one call, computed the same way on host and device.
//   persistent: unit descriptors, picks, weights, f16 tokens, slot mbarriers
//   region A:   phase 1-2 (tokens, router rows, plan, ranking)  |  the ring
//   region B:   gate/up partial tiles  |  down staging (activations, partials)
struct LayerLayout {
    size_t sd, ids, wts, xg, bars, last;
    size_t xs, wr, plan, topk, rk;
    size_t ring;
    size_t red, ah, al, ps;
    size_t gl;       // offset of the up matrix in a gate/up piece (bound of one tile)
    size_t du;       // bytes per unit in a down piece
    size_t slot;     // bytes per ring slot
    int ns;          // ring slots (0: the call does not fit)
    int m;           // units per down piece
    size_t total;
};

__host__ __device__ inline LayerLayout layer_layout(int fmt, int E, int K, int k, int H, int I, int T,
                                                    int has_shared, int rows) {
    LayerLayout L;
    const int n_ids = T * k, U = (n_ids < E ? n_ids : E) + 1, P = n_ids + (has_shared ? T : 0);
    size_t o = 0;
    L.sd = o; o = align16(o + (size_t)U * sizeof(UnitDesc));
    L.ids = o; o = align16(o + (size_t)n_ids * 4);
    L.wts = o; o = align16(o + (size_t)n_ids * 4);
    L.xg = o; o = align16(o + (size_t)(T + 1) * (H + 8) * 2);
    L.bars = o; o = align16(o + (size_t)kMaxSlots * 8);
    L.last = o; o = align128(o + (size_t)kMaxSlots * 4);
    const size_t a0 = o;
    // phases 1-2: tokens, router rows, plan, ranking
    size_t p = a0;
    L.xs = p; p = align16(p + (size_t)T * H * 2);
    L.wr = p; p = align16(p + (size_t)rows * H * 2);
    L.plan = p; p = align16(p + plan_layout(nullptr, E, K, n_ids, U, P).bytes);
    L.topk = p; p = align16(p + (size_t)(T < kLayerRankWarps ? T : kLayerRankWarps) * topk_bytes_per_warp(E));
    // one token: the rank keys (E <= 256) or the warps' sorted lists, then the picks' lower bounds
    L.rk = p; p = align16(p + (size_t)(E > kLThreads / 32 * kMaxTopK ? E : kLThreads / 32 * kMaxTopK) * 8 +
                          (size_t)kMaxTopK * 8);
    const size_t phase12 = p - a0;
    // region B: gate/up partials, or the down staging
    const size_t ld = (size_t)I + 8;
    const size_t red_bytes = (size_t)2 * 8 * 2 * 128 * 4;
    const size_t act_bytes = align16((size_t)(P + 1) * ld * 2);
    const size_t ps_bytes = down_rows_work_bytes(I, P) - 2 * (size_t)(P + 1) * ld * 2;
    const size_t down_bytes = 2 * act_bytes + align16(ps_bytes);
    const size_t b_bytes = align128(red_bytes > down_bytes ? red_bytes : down_bytes);
    // the ring
    L.gl = tile_bytes_bound(fmt, H);
    L.du = align128(tile_bytes_bound(fmt, I));
    L.slot = align128(2 * L.gl > L.du ? 2 * L.gl : L.du);
    L.m = (int)(L.slot / L.du);
    const size_t avail = kLayerSmemLimit > a0 + b_bytes ? kLayerSmemLimit - a0 - b_bytes : 0;
    size_t ns = avail / L.slot;
    if (ns > (size_t)kMaxSlots) ns = kMaxSlots;
    L.ns = (int)ns;
    const size_t a_bytes = align128(phase12 > ns * L.slot ? phase12 : ns * L.slot);
    L.ring = a0;
    L.red = a0 + a_bytes;
    L.ah = L.red;
    L.al = L.ah + act_bytes;
    L.ps = L.al + act_bytes;
    L.total = L.red + b_bytes;
    if (L.total > kLayerSmemLimit) L.ns = 0;
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


// ---------------------------------------------------------------------------
// Slot ring: mbarriers and bulk copies (sm_90+ PTX).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(bar) : "memory");
}
// Arrives and adds `bytes` to the transaction count the phase waits for.
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for the phase of the given parity to complete; false if the wait
// gave up (time or poll limit).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (unsigned it = 0; it < kSlotMaxPolls; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kSlotTimeoutNs) break;
    }
    return false;
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
    return p;
}
// Bulk copy global -> this CTA's shared memory (16-byte aligned addresses,
// size a multiple of 16), completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// The byte ranges of row tile rt of a slot matrix (R rows, C cols): the codes
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
        len[1] = 0;
        return 1;
    }
}

// Lane's share of chunk kc of a 16-row tile staged in shared memory by
// tile_ranges (codes at `t`, scales at `t + len0`; `soff` is the block-FP8
// scale range's start within its first 16 bytes). Same fragments as
// load_chunk reads from the slot.
template <int FMT>
__device__ __forceinline__ void smem_chunk(const uint8_t* t, uint32_t len0, uint32_t soff, int kc, int lane,
                                           Chunk<FMT>& ch) {
    if constexpr (FMT == FMT_Q4_0 || FMT == FMT_NVFP4) {
        ch.q = *reinterpret_cast<const uint4*>(t + (size_t)kc * 512 + lane * 16);
        ch.sc = *reinterpret_cast<const uint2*>(t + len0 + (size_t)kc * 64 + (lane >> 2) * 8);
    } else if constexpr (FMT == FMT_FP8_B128) {
        const uint8_t* q = t + (size_t)kc * 1024 + lane * 32;
        ch.q0 = *reinterpret_cast<const uint4*>(q);
        ch.q1 = *reinterpret_cast<const uint4*>(q + 16);
        ch.sc = *reinterpret_cast<const float*>(t + len0 + soff + (size_t)(kc >> 1) * 4);
    } else {
        const uint8_t* q = t + (size_t)kc * 2048 + lane * 64;
#pragma unroll
        for (int i = 0; i < 4; ++i) ch.q[i] = *reinterpret_cast<const uint4*>(q + 16 * i);
    }
}

// Start of the block-FP8 scale range of row tile rt within its 16-byte
// rounded copy (0 for the other formats).
template <int FMT>
__device__ __forceinline__ uint32_t scale_soff(int R, int C, int rt) {
    if constexpr (FMT == FMT_FP8_B128) {
        const int nct = (C + 127) / 128;
        const uint64_t s0 = (uint64_t)R * C + (uint64_t)((rt * 16) / 128) * nct * 4;
        return (uint32_t)(s0 & 15ull);
    } else {
        return 0u;
    }
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

// The pieces a CTA streams through its ring, in order: its gate/up items
// (unit, row tile) it = b + G j, then for each of its output row tiles
// rt = b + G r the down rows of units u0 .. u0 + m - 1.
struct Pieces {
    int b, G, RT, n_units, n_gu, n_rt, dpr, n;
};

__device__ __forceinline__ Pieces make_pieces(int b, int G, int RT, int RTD, int n_units, int m) {
    Pieces q;
    q.b = b;
    q.G = G;
    q.RT = RT;
    q.n_units = n_units;
    const int n_items = n_units * RT;
    q.n_gu = n_items > b ? (n_items - 1 - b) / G + 1 : 0;
    q.n_rt = RTD > b ? (RTD - 1 - b) / G + 1 : 0;
    q.dpr = (n_units + m - 1) / m;
    q.n = q.n_gu + q.n_rt * q.dpr;
    return q;
}

// Issues piece i into slot i % ns: bulk copies of its resident bytes, with one
// arrival on the slot's mbarrier (missed units' bytes are not copied: their
// consumers read the host store or the slot directly). One thread.
template <int FMT>
__device__ __forceinline__ void issue_piece(int i, const Pieces& q, const LayerLayout& L, const UnitDesc* sd, uint8_t* smem, int H,
                            int I, uint64_t pol) {
    const int slot = i % L.ns;
    const uint32_t bar = smem_u32(smem + L.bars) + slot * 8;
    const uint32_t dst = smem_u32(smem + L.ring) + (uint32_t)(slot * L.slot);
    reinterpret_cast<int*>(smem + L.last)[slot] = i;
    const uint64_t mgu = matrix_stride(FMT, I, H);
    uint64_t off[2];
    uint32_t len[2];
    if (i < q.n_gu) {
        const int it = q.b + q.G * i, u = it / q.RT, rt = it - u * q.RT;
        const UnitDesc& d = sd[u];
        if (d.dst) {
            mbar_arrive(bar);
            return;
        }
        const int nr = tile_ranges<FMT>(I, H, rt, off, len);
        uint32_t total = 0;
        for (int r = 0; r < nr; ++r) total += len[r];
        mbar_arrive_tx(bar, 2 * total);
        for (int mat = 0; mat < 2; ++mat) {
            const uint8_t* src = reinterpret_cast<const uint8_t*>(d.src) + mat * mgu;
            uint32_t o = dst + (uint32_t)(mat * L.gl);
            for (int r = 0; r < nr; ++r) {
                bulk_g2s(o, src + off[r], len[r], bar, pol);
                o += len[r];
            }
        }
    } else {
        const int di = i - q.n_gu, r = di / q.dpr, u0 = (di - r * q.dpr) * L.m;
        const int rt = q.b + q.G * r;
        const int nr = tile_ranges<FMT>(H, I, rt, off, len);
        uint32_t per = 0;
        for (int j = 0; j < nr; ++j) per += len[j];
        uint32_t total = 0;
        for (int v = 0; v < L.m && u0 + v < q.n_units; ++v)
            if (!sd[u0 + v].dst) total += per;
        if (!total) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_tx(bar, total);
        for (int v = 0; v < L.m && u0 + v < q.n_units; ++v) {
            const UnitDesc& d = sd[u0 + v];
            if (d.dst) continue;
            const uint8_t* src = reinterpret_cast<const uint8_t*>(d.src) + 2 * mgu;
            uint32_t o = dst + (uint32_t)(v * L.du);
            for (int j = 0; j < nr; ++j) {
                bulk_g2s(o, src + off[j], len[j], bar, pol);
                o += len[j];
            }
        }
    }
}

// Waits for piece i in its slot: first until the piece has been issued into
// the slot (its index is the slot's last issue), then for the slot's mbarrier
// phase of that piece. The ring's rule: every consumer of a piece waits here
// before it (or anyone) refills the slot with the piece ns ahead, so a slot
// holds at most one piece in flight, and once piece i is the slot's last issue
// the barrier's current phase is piece i's and the parity wait cannot match an
// older phase. (Two consumer groups take alternate pieces, so with an odd
// number of slots a group reaches pieces whose slot the other group refills.)
// False if either wait gave up.
__device__ __forceinline__ bool ring_wait(const LayerLayout& L, uint8_t* smem, int i) {
    const int slot = i % L.ns;
    const volatile int* last = reinterpret_cast<const volatile int*>(smem + L.last);
    if (last[slot] != i) {
        const unsigned long long t0 = globaltimer_ns();
        for (unsigned it = 0; last[slot] != i; ++it)
            if (globaltimer_ns() - t0 > kSlotTimeoutNs || it > kSlotMaxPolls) return false;
    }
    return mbar_wait(smem_u32(smem + L.bars) + slot * 8, (uint32_t)((i / L.ns) & 1));
}

// Waits (bounded) for the last piece issued into every slot; used before the
// CTA exits so no copy is in flight into its shared memory.
__device__ __forceinline__ void drain_ring(const LayerLayout& L, uint8_t* smem, int n_issued_max) {
    if (threadIdx.x != 0) return;
    const int* last = reinterpret_cast<const int*>(smem + L.last);
    const uint32_t bars = smem_u32(smem + L.bars);
    for (int sl = 0; sl < L.ns; ++sl) {
        const int i = last[sl];
        if (i >= 0 && i < n_issued_max) mbar_wait(bars + sl * 8, (uint32_t)((i / L.ns) & 1));
    }
}


// The gate and up accumulators of one warp's share of a gate/up item.
struct GateUpAcc {
    float g[4], u[4];
};

// One gate/up item (16-row tile rt) of a missed unit, read from the mapped
// host store over the host link (Wg: gate; up follows at the matrix stride)
// and written through to its slot (Dg) as it is read, by one group of eight
// warps (gw: the warp in the group, gtid: the thread); plus the item's share
// of the record's down matrix, copied to the slot, so the whole record crosses
// the link in this pass. Two chunk loads per matrix (4-bit formats; one
// otherwise) and the first batch of the down share are in flight at once.
// Inlined: a call would make the caller save its live registers around it,
// and those saves, in local memory that misses the small L1 left beside the
// shared memory, cost the all-hit path more than the deeper pull gains.
template <int FMT>
__device__ __forceinline__ GateUpAcc pull_item(const uint8_t* Wg, uint8_t* Dg, int I, int H, int rt, int gtid,
                                               int gw, int lane, const uint16_t* brow) {
    GateUpAcc r;
    float (&ag)[4] = r.g;
    float (&au)[4] = r.u;
#pragma unroll
    for (int i = 0; i < 4; ++i) ag[i] = au[i] = 0.f;
    constexpr bool kNib = FMT == FMT_Q4_0 || FMT == FMT_NVFP4;
    constexpr int CIF = kNib ? 2 : 1;  // chunks in flight per matrix
    constexpr int DS = kNib ? 2 : (FMT == FMT_FP8_B128 ? 2 : 1);    // down-share vectors in flight
    const uint64_t mgu = matrix_stride(FMT, I, H);
    const uint8_t* Wu = Wg + mgu;
    uint8_t* Du = Dg + mgu;
    const int KC = H / 64, cpw = (KC + 7) / 8, RT = I / 16;
    // this item's share of the down matrix
    const uint64_t nvec = matrix_stride(FMT, H, I) / 16, per = (nvec + RT - 1) / RT;
    const uint64_t v0 = (uint64_t)rt * per, v1 = v0 + per < nvec ? v0 + per : nvec;
    const uint8_t* src = Wg + 2 * mgu;
    uint8_t* dst = Dg + 2 * mgu;
    uint4 dbuf[DS];
#pragma unroll
    for (int i = 0; i < DS; ++i) {
        const uint64_t vi = v0 + gtid + (uint64_t)i * 256;
        if (vi < v1) dbuf[i] = ldg_stream(src + vi * 16);
    }
    if (rt == 0) {
        copy_matrix_tail<FMT>(Wg, Dg, I, H, gtid, 256);
        copy_matrix_tail<FMT>(Wu, Du, I, H, gtid, 256);
    }
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
        for (int i = 0; i < CIF; ++i) {
            const int kc = gw * cpw + c0 + i;
            if (c0 + i < cpw && kc < KC) {
                uint32_t bb[1][4][2];
                load_b_row(brow, kc, lane, bb[0]);
                mma_chunk<FMT, 1>(cg[i], bb, ag);
                mma_chunk<FMT, 1>(cu[i], bb, au);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < DS; ++i) {
        const uint64_t vi = v0 + gtid + (uint64_t)i * 256;
        if (vi < v1) stg_stream(dst + vi * 16, dbuf[i]);
    }
    // the rest of the share, if the item's share is larger than one batch
    constexpr int kBatch = 4;
    for (uint64_t v = v0 + (uint64_t)DS * 256 + gtid; v < v1; v += 256ull * kBatch) {
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
    return r;
}

// A CTA whose wait gave up writes NaN over its share of the output (every
// G-th block of the CTA size), so a call that could not complete shows in its
// output, not only in the error bit moe_cache_stats reports.
__device__ __forceinline__ void poison_out(float* out, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) out[i] = __int_as_float(0x7fc00000);
}

// kOneToken: the instantiation for one token and at most kLThreads (512)
// experts, one per thread, with the many-token ranking left out (its
// registers would crowd the rest).
template <int FMT, bool kOneToken>
__global__ void __launch_bounds__(kLThreads, 1) k_layer(const __grid_constant__ CacheDev c, const __grid_constant__ Scratch s,
                                                      const __grid_constant__ RouteArgs a, float* __restrict__ out) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ unsigned long long clk;
    __shared__ int rerank;
    __shared__ int slot_err;
    __shared__ unsigned tmax[kLayerMaxTokens];  // largest |bf16| bits of each token (its fp16 prescale)
    __shared__ int psh[kLayerMaxPairs];         // the pairs' activation prescales
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const int E = c.E, H = c.H, I = c.I, k = c.k, T = kOneToken ? 1 : a.T;
    const int n_ids = T * k;
    const int U = min(n_ids, E) + 1;
    const int P = n_ids + (c.has_shared ? T : 0);
    const int pool = c.pool_mode ? 0 : a.layer;
    // logits: warp w < 4 of CTA b < NL computes expert 4 b + w, so only the
    // first NL CTAs, which start first on the SMs the previous call frees,
    // gate the ranking
    const int rows = E < kLogitWarps ? E : kLogitWarps;
    const int NL = (E + kLogitWarps - 1) / kLogitWarps;
    // When the committing CTA owns no output row tile it commits after the
    // second barrier; then nothing is written that any CTA reads before it,
    // and the first barrier reduces to waiting for the logit CTAs.
    const bool logit_wait = G - 1 >= H / 16;
    // the layout lives in shared memory: its fields are read once per phase,
    // and held in registers they would be spilled
    __shared__ LayerLayout sL;
    if (threadIdx.x == 0) sL = layer_layout(FMT, E, c.K, k, H, I, T, c.has_shared, rows);
    __syncthreads();
    const LayerLayout& L = sL;
    UnitDesc* sd = reinterpret_cast<UnitDesc*>(smem + L.sd);
    int* sids = reinterpret_cast<int*>(smem + L.ids);
    float* swts = reinterpret_cast<float*>(smem + L.wts);
    uint16_t* xg = reinterpret_cast<uint16_t*>(smem + L.xg);
    const int ldx = H + 8;
    const uint32_t bars = smem_u32(smem + L.bars);
    if (tid < kMaxSlots) reinterpret_cast<int*>(smem + L.last)[tid] = -1;
    if (tid == 0) {
        for (int i = 0; i < L.ns; ++i) mbar_init(bars + i * 8, 1);
        fence_mbar_init();
        slot_err = 0;
    }

    // ---- 1. logits ---------------------------------------------------------
    // warp w < 4 of CTA b owns expert 4 b + w; its router row does not depend
    // on the preceding grid, so its copy to shared memory starts before the
    // wait (each lane copies, and later reads, its own 16-byte vectors)
    const int e_mine = warp < kLogitWarps ? b * kLogitWarps + warp : E;
    uint16_t* wr = reinterpret_cast<uint16_t*>(smem + L.wr) + (size_t)warp * H;
    if (e_mine < E)
        for (int i = 0; i < router_nvec(H) && lane * 8 + i * 256 < H; ++i)
            cp_async16(wr + lane * 8 + i * 256, a.w + (size_t)e_mine * H + lane * 8 + i * 256);
    const PlanSmem m = plan_layout(smem + L.plan, E, c.K, n_ids, U, P);
    // the pool's state (stamps, keys, the layer's slot map, its clock, NVFP4
    // global scales): read by every CTA before the first barrier, written
    // only by the committing CTA after it; read before the wait on the
    // preceding grid when that grid cannot be writing it
    auto stage_state = [&]() {
        const unsigned long long* lu = c.last_use + (size_t)pool * c.K;
        const int* kof = c.key_of + (size_t)pool * c.K;
        const int* smap = c.slot_map + (size_t)a.layer * E;
        for (int i = tid; i < c.K; i += kLThreads) {
            cp_async8(m.lu + i, lu + i);
            cp_async4(m.kof + i, kof + i);
        }
        for (int i = tid; i < E; i += kLThreads) cp_async4(m.smap + i, smap + i);
        if (c.fmt == FMT_NVFP4) {
            for (int i = tid; i < E * 3; i += kLThreads) cp_async4(m.gl + i, c.gtable + (size_t)a.layer * E * 3 + i);
            if (tid < 3) cp_async4(m.gl + E * 3 + tid, c.gtable + ((size_t)c.L * E + a.layer) * 3 + tid);
        }
        if (tid == 0) cp_async8(&clk, c.clock + pool);
    };
    if (a.early) stage_state();
    griddep_wait();
    griddep_launch();
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L.xs);
    unsigned phase = 0, call_par = 0;
    {
        // the tokens, and the pool's state if not staged yet
        // two groups: the tokens (with the router rows and any early state),
        // which the logits wait for, and the state, which only the ranking
        // and the plan need
        for (int i = tid; i < T * (H / 8); i += kLThreads) cp_async16(xs + (size_t)i * 8, a.x + (size_t)i * 8);
        cp_async_commit();
        if (!a.early) stage_state();
        cp_async_commit();
        if (tid < kLayerMaxTokens) tmax[tid] = 0u;
        // the pairs' activation maxima start from zero; this is ordered before
        // every other CTA's gate/up by the logit announcement (or the grid
        // barrier) below, and after the previous call's readers by the wait
        if (b == 0) {
            for (int i = tid; i < P; i += kLThreads) s.act_amax[i] = 0u;
        }
        for (int i = tid; i < E; i += kLThreads) m.first[i] = 0x7fffffff;
        for (int i = tid; i <= E / 32; i += kLThreads) m.missbits[i] = 0u;
        if (tid == 0) {
            rerank = 0;
            unsigned cur;
            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];\n" : "=r"(cur) : "l"(s.grid_bar) : "memory");
            phase = cur & 0x80000000u;
            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];\n" : "=r"(cur) : "l"(s.pass_ctr + 1) : "memory");
            call_par = cur & 1u;
        }
        cp_async_wait_but_last();
        __syncthreads();
    }
    // the logits first, announced as soon as they are written: they gate
    // every CTA's ranking, the f16 copy below only this CTA's expert phase
    if (e_mine < E)
        for (int t = 0; t < T; ++t) router_logit_row(c, a, xs + (size_t)t * H, wr, t, e_mine, s.logits, s.bounds);
    // thread 0: this call's parity, which alternates from call to call (the
    // last CTA past the logit wait flips it for the next call)
    const unsigned parity = call_par;
    if (logit_wait && b < NL) {
        __syncthreads();
        if (tid == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;\n" ::"l"(s.logit_ctr + parity) : "memory");
    }
    {
        // f16 copy of the tokens for the expert B operand (converted as the
        // gate/up kernel does, with each token's power-of-two prescale, taken
        // from the token's largest magnitude as the routing kernel takes it);
        // row T is zero
        if constexpr (FMT != FMT_BF16) {
            for (int t = 0; t < T; ++t) {
                unsigned mx = 0u;
                for (int v = tid; v < H / 8; v += kLThreads) {
                    const uint4 val = *reinterpret_cast<const uint4*>(xs + (size_t)t * H + v * 8);
                    mx = max(mx, max(max(bf16x2_absmax(val.x), bf16x2_absmax(val.y)),
                                     max(bf16x2_absmax(val.z), bf16x2_absmax(val.w))));
                }
                mx = __reduce_max_sync(0xffffffffu, mx);
                if (lane == 0 && mx) atomicMax(&tmax[t], mx);
            }
            __syncthreads();
        }
        for (int i = tid; i < T * (H / 8); i += kLThreads) {
            const int t = i / (H / 8), v = i - t * (H / 8);
            const uint4 val = *reinterpret_cast<const uint4*>(xs + (size_t)i * 8);
            uint32_t w4[4] = {val.x, val.y, val.z, val.w};
            if constexpr (FMT != FMT_BF16) {
                const float sc = pow2f(-token_shift(tmax[t]));
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float lo = __uint_as_float(w4[j] << 16) * sc;
                    const float hi = __uint_as_float(w4[j] & 0xffff0000u) * sc;
                    w4[j] = h2_as_u32(__floats2half2_rn(lo, hi));
                }
            }
            *reinterpret_cast<uint4*>(xg + (size_t)t * ldx + v * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        for (int i = tid; i < ldx / 2; i += kLThreads) reinterpret_cast<uint32_t*>(xg + (size_t)T * ldx)[i] = 0u;
    }
    cp_async_wait();  // the pool's state (made visible by the barriers below)
    if (logit_wait) {
        // every CTA waits until all NL logit CTAs have announced theirs
        __shared__ int lw_ok;
        __syncthreads();
        if (tid == 0) {
            const unsigned* ctr = s.logit_ctr + parity;
            const unsigned long long t0 = globaltimer_ns();
            int good = 1;
            for (unsigned it = 0;; ++it) {
                unsigned cur;
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(cur) : "l"(ctr) : "memory");
                if (cur >= (unsigned)NL) break;
                if (globaltimer_ns() - t0 > kBarrierTimeoutNs || it > kBarrierMaxPolls) {
                    atomicOr(s.err, 1u);
                    good = 0;
                    break;
                }
            }
            lw_ok = good;
        }
        __syncthreads();
        if (!lw_ok) {  // nothing is in flight yet
            poison_out(out, T * H);
            return;
        }
        // the last CTA past the wait clears this parity's counter for the call
        // two ahead and flips the parity for the next call
        if (tid == 0 && atomicAdd(s.pass_ctr, 1u) == (unsigned)G - 1) {
            s.logit_ctr[parity] = 0u;
            s.pass_ctr[0] = 0u;
            s.pass_ctr[1] = parity ^ 1u;
        }
    } else if (!grid_barrier(s.grid_bar, s.err, phase)) {
        poison_out(out, T * H);  // nothing is in flight yet
        return;
    }

    // ---- 2. top-k and plan in every CTA ----------------------------------
    if (kOneToken) {
        // one token: every expert's key held by its own thread, ranked by
        // counting (up to 256 experts) or by a threshold selection
        const TopkSmem tw = topk_layout(smem + L.topk, E);
        if (E <= 256)
            topk_rank_block(c, s, a, tw, reinterpret_cast<unsigned long long*>(smem + L.rk),
                            reinterpret_cast<float2*>(smem + L.rk + (size_t)E * 8), &rerank, sids, swts);
        else
            topk_block_select(c, s, a, tw, reinterpret_cast<unsigned long long*>(smem + L.rk),
                              reinterpret_cast<float2*>(smem + L.rk + (size_t)(kLThreads / 32) * kMaxTopK * 8),
                              &rerank, sids, swts);
    } else {
        const int nrw = min(T, kLayerRankWarps);
        if (warp < nrw) {
            const TopkSmem tw = topk_layout(smem + L.topk + (size_t)warp * topk_bytes_per_warp(E), E);
            for (int t = warp; t < T; t += nrw) topk_dispatch(c, s, a, t, tw, &rerank, sids, swts);
        }
    }
    __syncthreads();
    // The last CTA commits the call's cache transaction. When it owns no output
    // row tile it commits after the second barrier, off the critical path: it
    // takes the same descriptors as the others before, and runs the full plan
    // on a fresh copy of the pool's state after (nothing else writes that state
    // during the call, and every CTA read it before the first barrier).
    const bool commit = b == G - 1;
    const bool defer = commit && logit_wait;
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
    // A single token whose picks are all resident needs no cache transaction
    // to find its weights: unit j is pick j, read in place from its slot (the
    // descriptors the full plan gives such a call). The committing CTA still
    // runs the full plan, which also touches the slots and counts the hits.
    // A single token with misses needs only the victims beyond that: unit j is
    // still pick j; the hits are stamped in pick order as the full plan stamps
    // them, and miss i in ascending expert order takes victim i (the full
    // plan's first steps for one token, without its general dedupe and pair
    // lists).
    __shared__ int fast;  // 1: every pick resident; 2: one token with misses
    if (warp == 0) {
        int ok = 0;
        if (T == 1 && (!commit || defer)) {
            const int sl = lane < k ? m.smap[sids[lane]] : 0;
            ok = __all_sync(0xffffffffu, sl >= 0);
            if (!ok) {
                const unsigned hb = __ballot_sync(0xffffffffu, lane < k && sl >= 0);
                if (lane < k && sl >= 0) m.lu[sl] = clk + __popc(hb & ((1u << lane) - 1u));
                const int nmiss = k - __popc(hb);
                if (lane == 0) m.scal[1] = nmiss;
                ok = nmiss <= kVictimLists && c.K <= 64 * kLThreads ? 2 : 0;
            } else if (lane <= k) {
                UnitDesc d;
                d.pstart = 0;
                d.np = 1;
#pragma unroll
                for (int j = 1; j < 8; ++j) d.pair8[j] = -1;
                d.pair8[0] = lane;
                d.dst = 0;
                d.hit = 1;
                if (lane < k) {
                    const int e = sids[lane];
                    d.expert = e;
                    d.slot = sl;
                    d.src = (uint64_t)(c.pool + ((size_t)pool * c.K + sl) * c.slot_stride);
                    for (int j = 0; j < 3; ++j) d.g[j] = c.fmt == FMT_NVFP4 ? m.gl[e * 3 + j] : 1.0f;
                } else {
                    d.expert = -1;
                    d.slot = -1;
                    d.src = (uint64_t)(c.shared_w + (size_t)a.layer * c.slot_stride);
                    for (int j = 0; j < 3; ++j) d.g[j] = c.fmt == FMT_NVFP4 ? m.gl[E * 3 + j] : 1.0f;
                }
                if (lane < k || c.has_shared) sd[lane] = d;
            }
        }
        if (lane == 0) fast = ok;
    }
    __syncthreads();
    int n_units;
    if (fast == 2) {
        const int nmiss = m.scal[1];
        if (c.lfu) lfu_victim_keys(c, m, clk);
        select_victims(m, c.K, nmiss);
        if (warp == 0 && lane <= k) {
            UnitDesc d;
            d.pstart = 0;
            d.np = 1;
#pragma unroll
            for (int j = 1; j < 8; ++j) d.pair8[j] = -1;
            d.pair8[0] = lane;
            d.dst = 0;
            d.hit = 1;
            if (lane < k) {
                const int e = sids[lane];
                const int sl = m.smap[e];
                d.expert = e;
                for (int j = 0; j < 3; ++j) d.g[j] = c.fmt == FMT_NVFP4 ? m.gl[e * 3 + j] : 1.0f;
                if (sl >= 0) {
                    d.slot = sl;
                    d.src = (uint64_t)(c.pool + ((size_t)pool * c.K + sl) * c.slot_stride);
                } else {
                    int r = 0;  // this miss's place among the misses, ascending expert
                    for (int j = 0; j < k; ++j) r += (m.smap[sids[j]] < 0 && sids[j] < e) ? 1 : 0;
                    const int v = m.victims[r];
                    d.slot = v;
                    d.hit = 0;
                    d.src = (uint64_t)(c.store + ((size_t)a.layer * E + e) * c.slot_stride);
                    d.dst = (uint64_t)(c.pool + ((size_t)pool * c.K + v) * c.slot_stride);
                }
            } else {
                d.expert = -1;
                d.slot = -1;
                d.src = (uint64_t)(c.shared_w + (size_t)a.layer * c.slot_stride);
                for (int j = 0; j < 3; ++j) d.g[j] = c.fmt == FMT_NVFP4 ? m.gl[E * 3 + j] : 1.0f;
            }
            if (lane < k || c.has_shared) sd[lane] = d;
        }
        n_units = k + (c.has_shared ? 1 : 0);
    } else if (fast) {
        n_units = k + (c.has_shared ? 1 : 0);
    } else {
        plan_small(c, s, a, m, clk, sids, sd, commit && !defer);
        n_units = m.scal[0] + (c.has_shared ? 1 : 0);
    }
    __syncthreads();  // the ring below overlaps the plan's shared memory

    // ---- 3. stream the call's weight bytes; gate/up + SwiGLU ---------------
    const int RT = I / 16, KC = H / 64, RTD = H / 16, KCD = I / 64;
    const uint64_t mgu = matrix_stride(FMT, I, H);
    const Pieces q = make_pieces(b, G, RT, RTD, n_units, L.m);
    const uint64_t pol = policy_evict_first();
    // The ring's first fill: piece p < n0 goes into slot p. The first piece of
    // each group is requested now; piece p >= 2 when its group's item p - 2
    // has landed, so the first pieces do not queue behind the whole fill and
    // the groups start computing while the rest streams in (a piece no gate/up
    // item of its group precedes is requested now too).
    const int n0 = min(q.n, L.ns);
    if (lane == 0 && warp < n0 && (warp < 2 || warp - 2 >= q.n_gu)) {
        // lane 0 of warp w issues piece w; the ring reuses shared memory the
        // generic proxy wrote in phases 1-2
        fence_proxy_async();
        issue_piece<FMT>(warp, q, L, sd, smem, H, I, pol);
    }
    const uint8_t* ring = smem + L.ring;
    {
        // group g (warps 8g .. 8g+7) takes items j = g, g + 2, ...; the K split
        // over the group's warps and the warp-ordered sum are the gate/up
        // kernel's
        const int grp = warp >> 3, gw = warp & 7, gtid = tid & 255;
        float* red = reinterpret_cast<float*>(smem + L.red) + (size_t)grp * 8 * 2 * 128;
        const int cpw = (KC + 7) / 8;
        for (int j = grp; j < q.n_gu; j += 2) {
            const int it = b + G * j, u = it / RT, rt = it - u * RT;
            const UnitDesc d = sd[u];
            const int slot = j % L.ns;
            const uint8_t* Wg = reinterpret_cast<const uint8_t*>(d.src);
            uint8_t* Dg = d.dst ? reinterpret_cast<uint8_t*>(d.dst) : nullptr;
            const int np = d.np;
            // this lane's token row of the B tile (zero row past the unit's pairs)
            const int col = lane & 7;
            const int tok = col < np ? pair_token(pair_at(s, d, col), T, k) : T;
            const uint16_t* brow = xg + (size_t)tok * ldx;
            float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
            // every item waits for its piece, a missed unit's too (whose piece
            // carries no bytes): the group refills the slot after the item, and
            // a slot may only be refilled once its current piece has been
            // issued, that is once the piece before it was consumed
            if (!ring_wait(L, smem, j)) slot_err = 1;
            if (gtid == 0 && j + 2 < n0) {  // the group's piece two ahead, of the first fill
                fence_proxy_async();
                issue_piece<FMT>(j + 2, q, L, sd, smem, H, I, pol);
            }
            if (!Dg) {
                // resident: the tile is in slot j % ns
                const uint8_t* pg = ring + (size_t)slot * L.slot;
                const uint8_t* pu = pg + L.gl;
                const uint32_t len0 = (uint32_t)KC * (FMT == FMT_BF16 ? 2048 : (FMT == FMT_FP8_B128 ? 1024 : 512));
                const uint32_t soff = scale_soff<FMT>(I, H, rt);
                for (int c0 = 0; c0 < cpw; ++c0) {
                    const int kc = gw * cpw + c0;
                    if (kc >= KC) break;
                    Chunk<FMT> cg, cu;
                    smem_chunk<FMT>(pg, len0, soff, kc, lane, cg);
                    smem_chunk<FMT>(pu, len0, soff, kc, lane, cu);
                    uint32_t bb[1][4][2];
                    load_b_row(brow, kc, lane, bb[0]);
                    mma_chunk<FMT, 1>(cg, bb, ag);
                    mma_chunk<FMT, 1>(cu, bb, au);
                }
            } else {
                // missed: read the tile from the mapped host store over the
                // host link and write it through to the slot
                if (gtid == 0) atomicMin(s.copy_t0, globaltimer_ns());
                const GateUpAcc r = pull_item<FMT>(Wg, Dg, I, H, rt, gtid, gw, lane, brow);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    ag[i] = r.g[i];
                    au[i] = r.u[i];
                }
            }
            const int g = lane >> 2, qd = lane & 3;
            float* rg = red + (size_t)(gw * 2) * 128;
            float* ru = rg + 128;
            rg[g * 8 + 2 * qd] = ag[0];
            rg[g * 8 + 2 * qd + 1] = ag[1];
            rg[(g + 8) * 8 + 2 * qd] = ag[2];
            rg[(g + 8) * 8 + 2 * qd + 1] = ag[3];
            ru[g * 8 + 2 * qd] = au[0];
            ru[g * 8 + 2 * qd + 1] = au[1];
            ru[(g + 8) * 8 + 2 * qd] = au[2];
            ru[(g + 8) * 8 + 2 * qd + 1] = au[3];
            group_sync(grp);
            // the slot is consumed: refill it with the piece ns ahead
            if (gtid == 0 && j + L.ns < q.n) issue_piece<FMT>(j + L.ns, q, L, sd, smem, H, I, pol);
            if (gtid < 128) {
                const int row = gtid >> 3, cc = gtid & 7;
                float gs = 0.f, us = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    gs += red[(size_t)(w * 2) * 128 + gtid];
                    us += red[(size_t)(w * 2 + 1) * 128 + gtid];
                }
                const int pair = cc < np ? pair_at(s, d, cc) : -1;
                float av = 0.f;
                if (pair >= 0) {
                    const float up = FMT == FMT_BF16 ? 1.0f : pow2f(token_shift(tmax[pair_token(pair, T, k)]));
                    av = swiglu_scaled(gs, us, d.g[0], d.g[1], up);
                }
                store_act<FMT>(s, pair, I, rt * 16 + row, av);
            }
            if (Dg && gtid == 0) atomicMax(s.copy_t1, globaltimer_ns());
            group_sync(grp);
        }
    }
    // ---- 4. down projection + combine by row tiles -------------------------
    uint16_t* ah = reinterpret_cast<uint16_t*>(smem + L.ah);
    uint16_t* al = reinterpret_cast<uint16_t*>(smem + L.al);
    float* ps = reinterpret_cast<float*>(smem + L.ps);
    const int ld = I + 8;
    const int ncg = (KCD + kDRChunks - 1) / kDRChunks;
    const uint32_t len0 = (uint32_t)KCD * (FMT == FMT_BF16 ? 2048 : (FMT == FMT_FP8_B128 ? 1024 : 512));
    const int g = lane >> 2, qd = lane & 3;
    // one (unit, chunk group) item of row tile rt: the unit's partial sums over
    // its chunk group (pdv: the unit's down rows in the ring)
    auto down_item = [&](int u, int cgi, const uint8_t* pdv, int rt, uint32_t soff) {
        const UnitDesc& d = sd[u];
        const int col = lane & 7;
        const int pr = col < d.np ? d.pair8[col] : P;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ci = 0; ci < kDRChunks; ++ci) {
            const int kc = cgi * kDRChunks + ci;
            if (kc >= KCD) break;
            Chunk<FMT> ch;
            if (d.dst) {
                // a missed record: written to its slot by the gate/up pass
                load_chunk_cg<FMT>(reinterpret_cast<const uint8_t*>(d.dst) + 2 * mgu, H, I, rt, kc, lane, ch);
            } else {
                smem_chunk<FMT>(pdv, len0, soff, kc, lane, ch);
            }
            uint32_t bf[2][4][2];
            const uint16_t* rh = ah + (size_t)pr * ld + kc * 64 + (lane >> 3) * 8;
            const uint16_t* rl = al + (size_t)pr * ld + kc * 64 + (lane >> 3) * 8;
            ldmatrix_x4(bf[0][0][0], bf[0][0][1], bf[0][1][0], bf[0][1][1], rh);
            ldmatrix_x4(bf[0][2][0], bf[0][2][1], bf[0][3][0], bf[0][3][1], rh + 32);
            ldmatrix_x4(bf[1][0][0], bf[1][0][1], bf[1][1][0], bf[1][1][1], rl);
            ldmatrix_x4(bf[1][2][0], bf[1][2][1], bf[1][3][0], bf[1][3][1], rl + 32);
            mma_chunk<FMT, 2>(ch, bf, acc);
        }
        const float gd = d.g[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                const int cc = 2 * qd + c2;
                if (cc < d.np) {
                    const int pair = d.pair8[cc];
                    ps[((size_t)cgi * P + pair) * 16 + g + 8 * h2] = acc[2 * h2 + c2] * gd * pow2f(psh[pair]);
                }
            }
        }
    };
    // the committing CTA runs the full plan on a fresh copy of the pool's state
    // (nothing else writes that state during the call, and every CTA read it
    // before the logit wait); its ring and staging are free once its own
    // gate/up is done
    auto deferred_plan = [&]() {
        stage_state();
        for (int i = tid; i < E; i += kLThreads) m.first[i] = 0x7fffffff;
        for (int i = tid; i <= E / 32; i += kLThreads) m.missbits[i] = 0u;
        cp_async_wait();
        __syncthreads();
        plan_small(c, s, a, m, clk, sids, sd, true);
    };
    auto book_copy_time = [&]() {
        // every miss of the call has been streamed: book the time
        const unsigned long long t1 = atomicAdd(s.copy_t1, 0ull);
        if (t1) {
            const unsigned long long t0 = atomicAdd(s.copy_t0, 0ull);
            c.stats[a.bucket * 5 + 4] += t1 - t0;
            *s.copy_t0 = ~0ull;
            *s.copy_t1 = 0ull;
        }
    };
    if (!grid_barrier(s.grid_bar, s.err, phase)) {
        __syncthreads();
        drain_ring(L, smem, q.n);
        poison_out(out, T * H);
        return;
    }
    if (defer) deferred_plan();
    if (commit && tid == 0) book_copy_time();
    if (q.n_rt > 0) {
        down_stage_act<FMT>(s, P, I, ah, al, psh);
        __syncthreads();
        for (int r = 0; r < q.n_rt; ++r) {
            const int rt = b + G * r;
            const uint32_t soff = scale_soff<FMT>(H, I, rt);
            if (q.n_rt * q.dpr <= L.ns) {
                // the down pieces take distinct slots, and each was issued by
                // the end of gate/up (at the start, or as the refill of a
                // gate/up piece), so no slot is refilled here: all units'
                // items in one pass, each waiting for its own piece
                for (int itm = warp; itm < n_units * ncg; itm += kLWarps) {
                    const int u = itm / ncg, cgi = itm - u * ncg, pc = u / L.m;
                    const int i = q.n_gu + r * q.dpr + pc;
                    if (!ring_wait(L, smem, i)) slot_err = 1;
                    down_item(u, cgi, ring + (size_t)(i % L.ns) * L.slot + (size_t)(u - pc * L.m) * L.du, rt, soff);
                }
                __syncthreads();
            } else {
                for (int pc = 0; pc < q.dpr; ++pc) {
                    const int i = q.n_gu + r * q.dpr + pc;
                    const int slot = i % L.ns;
                    if (!ring_wait(L, smem, i)) slot_err = 1;
                    const int u0 = pc * L.m;
                    const int nup = min(L.m, n_units - u0);
                    const uint8_t* pd = ring + (size_t)slot * L.slot;
                    for (int itm = warp; itm < nup * ncg; itm += kLWarps) {
                        const int v = itm / ncg, cgi = itm - v * ncg;
                        down_item(u0 + v, cgi, pd + (size_t)v * L.du, rt, soff);
                    }
                    __syncthreads();
                    // the slot is consumed: refill it with the piece ns ahead
                    if (tid == 0 && i + L.ns < q.n) issue_piece<FMT>(i + L.ns, q, L, sd, smem, H, I, pol);
                }
            }
            combine_rows(ps, swts, T, k, P, ncg, c.has_shared, out + (size_t)rt * 16, H);
            __syncthreads();
        }
    }
    __syncthreads();
    if (tid == 0 && slot_err) atomicOr(s.err, 2u);
    drain_ring(L, smem, q.n);
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
    if (P > kLayerMaxPairs || G <= 0 || (c.E + kLogitWarps - 1) / kLogitWarps > G) return 0;
    const LayerLayout L =
        layer_layout(c.fmt, c.E, c.K, c.k, c.H, c.I, T, c.has_shared, c.E < kLogitWarps ? c.E : kLogitWarps);
    return L.ns >= 1 && L.total <= kLayerSmemLimit ? L.total : 0;
}

template <int FMT, bool kOneToken>
static bool layer_launch_as(const CacheDev& c, const Scratch& s, const RouteArgs& a, float* out, size_t sm,
                            cudaStream_t st, bool pdl) {
    static size_t set = 0;
    if (sm > set) {
        if (cudaFuncSetAttribute(k_layer<FMT, kOneToken>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) !=
            cudaSuccess)
            return false;
        set = sm;
    }
    // one CTA per SM, all resident: the grid barriers rely on it
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_layer<FMT, kOneToken>, kLThreads, sm) !=
            cudaSuccess ||
        per_sm < 1)
        return false;
    // a cooperative launch (the runtime starts the grid only when every CTA can
    // be resident, which the grid-wide waits need), with programmatic
    // dependent launch first
    static int form = kCoopWithPdl;
    const dim3 grid(layer_ctas()), block(kLThreads);
    return launch_cooperative(form, pdl, [&](bool with_pdl) {
        if (launch_ex_coop(k_layer<FMT, kOneToken>, grid, block, sm, st, with_pdl, true, c, s, a, out) ==
            cudaSuccess)
            return true;
        cudaGetLastError();
        return false;
    });
}

template <int FMT>
static bool layer_launch(const CacheDev& c, const Scratch& s, const RouteArgs& a, float* out, size_t sm,
                         cudaStream_t st, bool pdl) {
    if (a.T == 1 && c.E <= kLThreads) return layer_launch_as<FMT, true>(c, s, a, out, sm, st, pdl);
    return layer_launch_as<FMT, false>(c, s, a, out, sm, st, pdl);
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
