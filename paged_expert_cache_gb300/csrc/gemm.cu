// gemm.cu -- the expert FFN of a prefill call (T above the cache limit) as
// grouped GEMMs on the fifth-generation tensor cores (tcgen05, accumulators in
// tensor memory).
//
// A prefill call pushes a whole prompt through the layer at once, so each
// expert sees tens to hundreds of tokens: the work is a dense contraction
// per expert ("Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by
// streaming experts from NVMe" (atlasrepo.com), "Workflow": experts fetched
// in groups of 32 for the prompt; "Running a 95 GiB MoE Model on a 32 GiB
// GPU" (busyjay.com), "Prefill"). Per unit (a routed expert, or the shared
// expert) with its token pairs, the math is that of the decode kernels:
//   gate/up:  a[pair][i] = silu(g0 * (Wg x)_i) * (g1 * (Wu x)_i)
//   down:     part[pair][h] = g2 * (Wd a)_h
//   combine:  y[t] = sum_j w[t,j] part[t*k + j] (rank order) + part[shared]
// with Wg, Wu, Wd dequantised from the slot (or the staging arena) record.
//
// One CTA computes one (unit, 128-row tile, 128-pair tile) item: the weight
// rows are the M side of a 128 x 128 x 16 f16 MMA and the unit's token pairs
// the N side. Its eight warps dequantise the 64-column chunk of the weight
// tile into shared memory (K-major, 128-byte swizzle) and gather the pairs'
// token rows next to it; one thread issues the MMAs into tensor memory and
// commits them to an mbarrier, so the next chunk is staged while the tensor
// cores work on this one (two stages). The epilogue reads the accumulators
// with tcgen05.ld.
//
// Precision. Operands are fp16 with fp32 accumulation. NVFP4 weights are exact
// in fp16 (an E2M1 value times an E4M3 scale has at most five significant
// bits), and the per-matrix global scale is applied in the epilogue. Q4_0 and
// block-FP8 weights are rounded once to fp16 (relative error <= 2^-11). Tokens
// (bf16) enter as fp16 after the power-of-two prescale of their row (common.cuh),
// which keeps every value within 2^-32 of the row's largest exact, whatever
// the row's magnitude. The down projection takes each prescaled fp32
// activation as an fp16 hi + lo pair, two MMAs into one accumulator, as the
// decode kernels do. bf16 experts keep the mma.sync kernels (their operands
// would be bf16).
#include "expert_dev.cuh"

namespace moe {

constexpr int kGM = 128;          // weight rows per tile (M)
constexpr int kGN = 128;          // token pairs per tile (N)
constexpr int kGK = 64;           // K chunk: one 128-byte swizzle row of fp16
constexpr int kGThreads = 256;    // 8 warps; warp w stages row tile w (16 rows) of the M tile
constexpr int kGStages = 2;
constexpr uint32_t kGTile = (uint32_t)kGM * kGK * 2;  // 16 KB: one 128 x 64 fp16 tile
constexpr uint32_t kGStage = 3 * kGTile;               // A0, A1 / B-lo, B
constexpr uint32_t kGTmemCols = 256;                   // gate + up accumulators (down uses 128)
constexpr unsigned long long kGWaitNs = 200ull * 1000 * 1000;

// ---------------------------------------------------------------------------
// PTX wrappers: mbarriers, proxy fences, tcgen05.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t gsmem(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void gbar_init(uint32_t bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool gbar_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer_ns();
    for (unsigned it = 0; it < (1u << 26); ++it) {
        uint32_t ok;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if (globaltimer_ns() - t0 > kGWaitNs) break;
    }
    return false;
}
__device__ __forceinline__ void tc_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16, one CTA.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}
// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major tile in 128-byte swizzle atoms
// (8 rows x 128 bytes, 1024 bytes apart along M or N), starting at byte
// address `saddr` (the tile's atoms 1024-byte aligned; saddr may step by 32
// bytes inside the first row for the K16 slices).
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address
    d |= (uint64_t)1 << 16;                            // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;                  // stride byte offset: one 8-row atom
    d |= (uint64_t)1 << 46;                            // descriptor version
    d |= (uint64_t)2 << 61;                            // 128-byte swizzle
    return d;
}

// Instruction descriptor: fp32 accumulator, fp16 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t tc_idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Byte offset of fp16 element (r, c) (c < 64) in a K-major 128-byte swizzled
// tile: 16-byte chunk c/8 of row r sits at chunk (c/8) ^ (r % 8).
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((c >> 3) ^ r) & 7) << 4) + (c & 7) * 2);
}

// The GEMM's fp16 weights are the true ones divided by gemm_wscale (NVFP4: by
// 2^7, so one multiply builds them exactly); the epilogues multiply by it.
template <int FMT>
__host__ __device__ constexpr float gemm_wscale() { return FMT == FMT_NVFP4 ? 128.0f : 1.0f; }

// ---------------------------------------------------------------------------
// Weight fragments -> fp16 (fragment order of load_chunk: lane (g, q), k-step
// s holds (row g, cols 16s+2q..+1), (row g+8, same), (row g, cols 16s+2q+8..+9),
// (row g+8, same)), divided by gemm_wscale.
// ---------------------------------------------------------------------------
template <int FMT>
__device__ __forceinline__ void frag_to_f16(const Chunk<FMT>& ch, uint32_t (&a)[4][4]) {
    if constexpr (FMT == FMT_Q4_0) {
        const uint32_t w[4] = {ch.q.x, ch.q.y, ch.q.z, ch.q.w};
        const __half d[4] = {__low2half(u32_as_h2(ch.sc.x)), __high2half(u32_as_h2(ch.sc.x)),
                             __low2half(u32_as_h2(ch.sc.y)), __high2half(u32_as_h2(ch.sc.y))};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            uint32_t t[4];
            q4_to_frag(w[s], t);  // q - 8, exact
            const __half2 dg = __half2half2(d[s >> 1]), d8 = __half2half2(d[2 + (s >> 1)]);
            a[s][0] = h2_as_u32(__hmul2(u32_as_h2(t[0]), dg));
            a[s][1] = h2_as_u32(__hmul2(u32_as_h2(t[1]), d8));
            a[s][2] = h2_as_u32(__hmul2(u32_as_h2(t[2]), dg));
            a[s][3] = h2_as_u32(__hmul2(u32_as_h2(t[3]), d8));
        }
    } else if constexpr (FMT == FMT_NVFP4) {
        const uint32_t w[4] = {ch.q.x, ch.q.y, ch.q.z, ch.q.w};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            // code * 2^-14 (its bits) times scale * 2^7: the weight times 2^-7,
            // exact in fp16; the epilogues scale the sums back (gemm_wscale)
            const uint32_t scw = s < 2 ? ch.sc.x : ch.sc.y;
            const __half2 sh = __hmul2(u32_as_h2(e4m3x2_to_h2((scw >> (16 * (s & 1))) & 0xffffu)),
                                       __float2half2_rn(128.0f));
            const __half2 sg = __low2half2(sh), s8 = __high2half2(sh);
            a[s][0] = h2_as_u32(__hmul2(u32_as_h2(e2m1x2_bits_2m14(w[s])), sg));
            a[s][1] = h2_as_u32(__hmul2(u32_as_h2(e2m1x2_bits_2m14(w[s] >> 4)), s8));
            a[s][2] = h2_as_u32(__hmul2(u32_as_h2(e2m1x2_bits_2m14(w[s] >> 8)), sg));
            a[s][3] = h2_as_u32(__hmul2(u32_as_h2(e2m1x2_bits_2m14(w[s] >> 12)), s8));
        }
    } else if constexpr (FMT == FMT_FP8_B128) {
        const uint32_t w[8] = {ch.q0.x, ch.q0.y, ch.q0.z, ch.q0.w, ch.q1.x, ch.q1.y, ch.q1.z, ch.q1.w};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint32_t v[4] = {w[2 * s] & 0xffffu, w[2 * s] >> 16, w[2 * s + 1] & 0xffffu, w[2 * s + 1] >> 16};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float2 f = __half22float2(u32_as_h2(e4m3x2_to_h2(v[r])));
                a[s][r] = h2_as_u32(__floats2half2_rn(f.x * ch.sc, f.y * ch.sc));
            }
        }
    }
}

// Stores the fragments of row tile `w` (rows 16w .. 16w + 15 of the M tile).
__device__ __forceinline__ void store_frag(uint8_t* tile, int w, int lane, const uint32_t (&a)[4][4]) {
    const int g = lane >> 2, q = lane & 3;
    const int r0 = 16 * w + g, r1 = r0 + 8;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int c0 = 16 * s + 2 * q;
        *reinterpret_cast<uint32_t*>(tile + sw128(r0, c0)) = a[s][0];
        *reinterpret_cast<uint32_t*>(tile + sw128(r1, c0)) = a[s][1];
        *reinterpret_cast<uint32_t*>(tile + sw128(r0, c0 + 8)) = a[s][2];
        *reinterpret_cast<uint32_t*>(tile + sw128(r1, c0 + 8)) = a[s][3];
    }
}

// One work item: unit u, 128-pair tile n (blockIdx.y is the M tile).
struct GemmItem {
    int u, n;
};

// ---------------------------------------------------------------------------
// Work list of one launch: every (unit, pair tile) of the units the launch
// covers (map_unit: resident units + shared, or staging group `group`), in
// unit order. One CTA.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_gemm_items(CacheDev c, Scratch s, int kind, int group, int G, int Y,
                                                     int2* items, int* count) {
    __shared__ int wsum[32];
    __shared__ int base;
    griddep_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) base = 0;
    __syncthreads();
    for (int y0 = 0; y0 < Y; y0 += 1024) {
        const int y = y0 + tid;
        const int u = y < Y ? map_unit(s.plan, c.has_shared, kind, group, G, y) : -1;
        const int nt = u >= 0 ? (s.units[u].np + kGN - 1) / kGN : 0;
        int incl = nt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int v = wsum[lane], iv = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, iv, off);
                if (lane >= off) iv += o;
            }
            wsum[lane] = iv - v;  // exclusive prefix of the warps
        }
        __syncthreads();
        const int start = base + wsum[warp] + incl - nt;
        for (int n = 0; n < nt; ++n) items[start + n] = make_int2(u, n);
        __syncthreads();
        if (tid == 1023) base = start + nt;
        __syncthreads();
    }
    if (tid == 0) *count = base;
}

// ---------------------------------------------------------------------------
// Gate/up + SwiGLU.
// ---------------------------------------------------------------------------
template <int FMT>
__global__ void __launch_bounds__(kGThreads, 1) k_gemm_gateup(CacheDev c, Scratch s, const uint16_t* __restrict__ x,
                                                               int T, const int2* __restrict__ items,
                                                               const int* __restrict__ count) {
    extern __shared__ uint8_t gsm_raw[];
    __shared__ __align__(8) unsigned long long bars[kGStages];
    __shared__ uint32_t tmem_base;
    __shared__ int tok[kGN];
    __shared__ int pairs[kGN];
    __shared__ int tsh[kGN];  // each column's token prescale (token_shift)
    griddep_wait();
    if ((int)blockIdx.x >= *count) return;
    const int2 it = items[blockIdx.x];
    const UnitDesc d = s.units[it.x];
    const int n0 = it.y * kGN, m = blockIdx.y;
    const int nn = min(kGN, d.np - n0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = c.H, I = c.I, k = c.k, KC = H / 64;
    // 1024-byte aligned stages
    const uint32_t raw = gsmem(gsm_raw);
    uint8_t* sm = gsm_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sm_addr = gsmem(sm);
    if (warp == 0) {
        tc_alloc(gsmem(&tmem_base), kGTmemCols);
        tc_relinquish();
    }
    if (tid < kGStages) gbar_init(gsmem(&bars[tid]));
    if (tid < kGN) {
        const int p = tid < nn ? s.unit_pairs[d.pstart + n0 + tid] : -1;
        pairs[tid] = p;
        tok[tid] = p >= 0 ? pair_token(p, T, k) : -1;
        tsh[tid] = p >= 0 ? __ldg(s.tok_shift + tok[tid]) : 0;
    }
    if (tid == 0) asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint64_t mgu = matrix_stride(FMT, I, H);
    const uint8_t* Wg = reinterpret_cast<const uint8_t*>(d.src);
    const uint8_t* Wu = Wg + mgu;
    constexpr uint32_t idesc = tc_idesc_f16(kGM, kGN);
    bool ok = true;
    // Software pipeline: the global loads of chunk kc + 1 (weight fragments
    // and token rows) are issued before chunk kc is dequantised and stored,
    // so their latency overlaps the stores, the barrier and the MMA issue.
    // warp w dequantises row tile w of the gate and up tiles; thread i stages
    // token rows j = i / 8 + 32 r, 16-byte column chunk i % 8, r = 0..3
    constexpr int kTokPerThread = kGN * 8 / kGThreads;
    const int rt = m * (kGM / 16) + warp;
    // the item's whole weight tiles into L2 first: the register pipeline below
    // holds one chunk in flight, and its loads then wait on L2, not HBM
    if (warp == 0) {
        prefetch_rows<FMT>(Wg, I, H, m * (kGM / 16), kGM / 16, lane, 32);
        prefetch_rows<FMT>(Wu, I, H, m * (kGM / 16), kGM / 16, lane, 32);
    }
    Chunk<FMT> cg, cu;
    uint4 xv[kTokPerThread];
    auto load_next = [&](int kc) {
        load_chunk<FMT>(Wg, nullptr, I, H, rt, kc, lane, cg);
        load_chunk<FMT>(Wu, nullptr, I, H, rt, kc, lane, cu);
#pragma unroll
        for (int r = 0; r < kTokPerThread; ++r) {
            const int i = tid + r * kGThreads, j = i >> 3, cc = i & 7;
            xv[r] = tok[j] >= 0 ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)tok[j] * H + kc * 64 + cc * 8))
                                : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    load_next(0);
    for (int kc = 0; kc < KC; ++kc) {
        const int st = kc & 1;
        uint8_t* stage = sm + (size_t)st * kGStage;
        // the MMAs of chunk kc - 2 read this stage
        if (kc >= kGStages && !gbar_wait(gsmem(&bars[st]), (uint32_t)(((kc - kGStages) / kGStages) & 1))) ok = false;
        {
            uint32_t a[4][4];
            frag_to_f16<FMT>(cg, a);
            store_frag(stage, warp, lane, a);
            frag_to_f16<FMT>(cu, a);
            store_frag(stage + kGTile, warp, lane, a);
        }
        // tokens: bf16 -> fp16 with the token's power-of-two prescale (exact)
#pragma unroll
        for (int r = 0; r < kTokPerThread; ++r) {
            const int i = tid + r * kGThreads, j = i >> 3, cc = i & 7;
            const float sc = pow2f(-tsh[j]);
            uint32_t w4[4] = {xv[r].x, xv[r].y, xv[r].z, xv[r].w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
                w4[q] = h2_as_u32(__floats2half2_rn(__uint_as_float(w4[q] << 16) * sc,
                                                    __uint_as_float(w4[q] & 0xffff0000u) * sc));
            *reinterpret_cast<uint4*>(stage + 2 * kGTile + sw128(j, cc * 8)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        if (kc + 1 < KC) load_next(kc + 1);
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t a0 = sm_addr + st * kGStage, a1 = a0 + kGTile, b0 = a0 + 2 * kGTile;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint32_t acc = (kc | ks) != 0;
                tc_mma(tmem, tc_sdesc(a0 + 32 * ks), tc_sdesc(b0 + 32 * ks), idesc, acc);
                tc_mma(tmem + kGN, tc_sdesc(a1 + 32 * ks), tc_sdesc(b0 + 32 * ks), idesc, acc);
            }
            tc_commit(gsmem(&bars[st]));
        }
    }
    // the last commit covers every MMA of the item
    {
        const int last = KC - 1;
        if (!gbar_wait(gsmem(&bars[last & 1]), (uint32_t)((last / kGStages) & 1))) ok = false;
        // drain the other stage's commit too, so no arrival is pending at exit
        if (KC >= 2 && !gbar_wait(gsmem(&bars[(last - 1) & 1]), (uint32_t)(((last - 1) / kGStages) & 1))) ok = false;
    }
    tc_fence_after();
    // epilogue: warp w reads lanes 32 (w % 4) .. + 31 (rows of the M tile) and
    // columns (pairs) 64 (w / 4) .. + 63 of both accumulators
    {
        const int lq = warp & 3, half = warp >> 2;
        const int row = 32 * lq + lane;
        const int i_out = m * kGM + row;
#pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {
            const int col = 64 * half + 32 * cb;
            uint32_t g[32], u[32];
            tc_ld32(tmem + ((uint32_t)(32 * lq) << 16) + col, g);
            tc_ld32(tmem + ((uint32_t)(32 * lq) << 16) + kGN + col, u);
            tc_ld_wait();
            unsigned mx[32];  // |a| bits of this lane's row, per column
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int p = pairs[col + j];
                mx[j] = 0u;
                if (p >= 0) {
                    const float av = swiglu_scaled(__uint_as_float(g[j]), __uint_as_float(u[j]),
                                                   d.g[0] * gemm_wscale<FMT>(), d.g[1] * gemm_wscale<FMT>(),
                                                   pow2f(tsh[col + j]));
                    s.act[(size_t)p * I + i_out] = av;
                    mx[j] = __float_as_uint(fabsf(av));
                }
            }
            // the largest |a| of each column over the warp's 32 rows, for the
            // down projection's prescale: a transposing butterfly halves the
            // columns a lane keeps at each step and leaves column `lane` in mx[0]
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const bool upper = (lane & off) != 0;
#pragma unroll
                for (int cc = 0; cc < off; ++cc) {
                    const unsigned send = upper ? mx[cc] : mx[cc + off];
                    const unsigned keep = upper ? mx[cc + off] : mx[cc];
                    mx[cc] = max(keep, __shfl_xor_sync(0xffffffffu, send, off));
                }
            }
            if (pairs[col + lane] >= 0 && mx[0]) atomicMax(s.act_amax + pairs[col + lane], mx[0]);
        }
    }
    if (!ok && tid == 0) atomicOr(s.err, 4u);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(tmem, kGTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Down projection: part[pair][h] = g2 * (Wd a_pair)_h.
// ---------------------------------------------------------------------------
template <int FMT>
__global__ void __launch_bounds__(kGThreads, 1) k_gemm_down(CacheDev c, Scratch s, const int2* __restrict__ items,
                                                             const int* __restrict__ count) {
    extern __shared__ uint8_t gsm_raw[];
    __shared__ __align__(8) unsigned long long bars[kGStages];
    __shared__ uint32_t tmem_base;
    __shared__ int pairs[kGN];
    __shared__ int psh[kGN];  // each column's activation prescale (act_shift)
    griddep_wait();
    if ((int)blockIdx.x >= *count) return;
    const int2 it = items[blockIdx.x];
    const UnitDesc d = s.units[it.x];
    const int n0 = it.y * kGN, m = blockIdx.y;
    const int nn = min(kGN, d.np - n0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = c.H, I = c.I, KC = I / 64;
    const uint32_t raw = gsmem(gsm_raw);
    uint8_t* sm = gsm_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sm_addr = gsmem(sm);
    if (warp == 0) {
        tc_alloc(gsmem(&tmem_base), kGTmemCols);
        tc_relinquish();
    }
    if (tid < kGStages) gbar_init(gsmem(&bars[tid]));
    if (tid < kGN) {
        const int p = tid < nn ? s.unit_pairs[d.pstart + n0 + tid] : -1;
        pairs[tid] = p;
        psh[tid] = p >= 0 ? act_shift(__ldcg(s.act_amax + p)) : 0;
    }
    if (tid == 0) asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint8_t* Wd = reinterpret_cast<const uint8_t*>(d.src) + 2 * matrix_stride(FMT, I, H);
    constexpr uint32_t idesc = tc_idesc_f16(kGM, kGN);
    bool ok = true;
    // the same software pipeline as gate/up: chunk kc + 1's weight fragments
    // and activations are in flight while chunk kc is staged
    constexpr int kActPerThread = kGN * 8 / kGThreads;
    const int rt = m * (kGM / 16) + warp;
    if (warp == 0) prefetch_rows<FMT>(Wd, H, I, m * (kGM / 16), kGM / 16, lane, 32);  // as in gate/up
    Chunk<FMT> ch;
    float4 av[kActPerThread][2];
    auto load_next = [&](int kc) {
        load_chunk<FMT>(Wd, nullptr, H, I, rt, kc, lane, ch);
#pragma unroll
        for (int r = 0; r < kActPerThread; ++r) {
            const int i = tid + r * kGThreads, j = i >> 3, cc = i & 7;
            if (pairs[j] >= 0) {
                const float4* src = reinterpret_cast<const float4*>(s.act + (size_t)pairs[j] * I + kc * 64 + cc * 8);
                av[r][0] = __ldcg(src);
                av[r][1] = __ldcg(src + 1);
            } else {
                av[r][0] = av[r][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    };
    load_next(0);
    for (int kc = 0; kc < KC; ++kc) {
        const int st = kc & 1;
        uint8_t* stage = sm + (size_t)st * kGStage;
        if (kc >= kGStages && !gbar_wait(gsmem(&bars[st]), (uint32_t)(((kc - kGStages) / kGStages) & 1))) ok = false;
        {
            uint32_t a[4][4];
            frag_to_f16<FMT>(ch, a);
            store_frag(stage, warp, lane, a);
        }
        // activations of the pairs: fp32 -> fp16 hi (tile 2) + lo (tile 1)
#pragma unroll
        for (int r = 0; r < kActPerThread; ++r) {
            const int i = tid + r * kGThreads, j = i >> 3, cc = i & 7;
            uint4 hv = make_uint4(0u, 0u, 0u, 0u), lv = hv;
            {
                const float sc = pow2f(-psh[j]);  // the pair's prescale (exact)
                const float4 f0 = av[r][0], f1 = av[r][1];
                const float f[8] = {f0.x * sc, f0.y * sc, f0.z * sc, f0.w * sc,
                                    f1.x * sc, f1.y * sc, f1.z * sc, f1.w * sc};
                uint16_t h16[8], l16[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) split_hi_lo<FMT>(f[q], h16[q], l16[q]);
                uint32_t h[4], l[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    h[q] = (uint32_t)h16[2 * q] | ((uint32_t)h16[2 * q + 1] << 16);
                    l[q] = (uint32_t)l16[2 * q] | ((uint32_t)l16[2 * q + 1] << 16);
                }
                hv = make_uint4(h[0], h[1], h[2], h[3]);
                lv = make_uint4(l[0], l[1], l[2], l[3]);
            }
            *reinterpret_cast<uint4*>(stage + 2 * kGTile + sw128(j, cc * 8)) = hv;
            *reinterpret_cast<uint4*>(stage + kGTile + sw128(j, cc * 8)) = lv;
        }
        if (kc + 1 < KC) load_next(kc + 1);
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t a0 = sm_addr + st * kGStage, blo = a0 + kGTile, bhi = a0 + 2 * kGTile;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                tc_mma(tmem, tc_sdesc(a0 + 32 * ks), tc_sdesc(bhi + 32 * ks), idesc, (kc | ks) != 0);
                tc_mma(tmem, tc_sdesc(a0 + 32 * ks), tc_sdesc(blo + 32 * ks), idesc, 1u);
            }
            tc_commit(gsmem(&bars[st]));
        }
    }
    {
        const int last = KC - 1;
        if (!gbar_wait(gsmem(&bars[last & 1]), (uint32_t)((last / kGStages) & 1))) ok = false;
        if (KC >= 2 && !gbar_wait(gsmem(&bars[(last - 1) & 1]), (uint32_t)(((last - 1) / kGStages) & 1))) ok = false;
    }
    tc_fence_after();
    {
        const int lq = warp & 3, half = warp >> 2;
        const int row = 32 * lq + lane;
        const int h_out = m * kGM + row;
#pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {
            const int col = 64 * half + 32 * cb;
            uint32_t v[32];
            tc_ld32(tmem + ((uint32_t)(32 * lq) << 16) + col, v);
            tc_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int p = pairs[col + j];
                if (p >= 0)
                    s.part[(size_t)p * H + h_out] =
                        __uint_as_float(v[j]) * (d.g[2] * gemm_wscale<FMT>()) * pow2f(psh[col + j]);
            }
        }
    }
    if (!ok && tid == 0) atomicOr(s.err, 4u);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(tmem, kGTmemCols);
    }
}

// y[t][h] = sum_j w[t,j] part[t*k + j][h] in rank order, plus the shared
// expert's part (the combine of the decode kernels, over the whole prompt).
__global__ void k_combine(CacheDev c, Scratch s, float* __restrict__ out, int T) {
    griddep_wait();
    const int H = c.H, k = c.k;
    const size_t n = (size_t)T * H;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / H), h = (int)(i - (size_t)t * H);
        float y = 0.f;
        for (int j = 0; j < k; ++j) y = fmaf(s.wts[t * k + j], __ldcg(s.part + (size_t)(t * k + j) * H + h), y);
        if (c.has_shared) y += __ldcg(s.part + (size_t)(T * k + t) * H + h);
        out[i] = y;
    }
}

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------
static size_t gemm_smem() { return (size_t)kGStages * kGStage + 1024; }

template <int FMT>
static void gemm_fmt(const CacheDev& c, const Scratch& s, const uint16_t* x, int T, int kind, int group, int G,
                     int Y, int max_items, cudaStream_t st) {
    static bool set = false;
    if (!set) {
        cudaFuncSetAttribute(k_gemm_gateup<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm_smem());
        cudaFuncSetAttribute(k_gemm_down<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm_smem());
        set = true;
    }
    k_gemm_items<<<1, 1024, 0, st>>>(c, s, kind, group, G, Y, s.gemm_items, s.gemm_count);
    k_gemm_gateup<FMT><<<dim3(max_items, c.I / kGM), kGThreads, gemm_smem(), st>>>(c, s, x, T, s.gemm_items,
                                                                                  s.gemm_count);
    k_gemm_down<FMT><<<dim3(max_items, c.H / kGM), kGThreads, gemm_smem(), st>>>(c, s, s.gemm_items, s.gemm_count);
}

bool gemm_supported(const CacheDev& c) {
    return c.fmt != FMT_BF16 && c.I % kGM == 0 && c.H % kGM == 0;
}

size_t gemm_max_items(int P, int Y) { return (size_t)(P + kGN - 1) / kGN + (size_t)Y + 1; }

void launch_gemm(const CacheDev& c, const Scratch& s, const uint16_t* x, int T, int kind, int group, int G, int Y,
                 cudaStream_t st) {
    const int P = T * c.k + (c.has_shared ? T : 0);
    const int max_items = (int)gemm_max_items(P, Y);
    switch (c.fmt) {
    case FMT_Q4_0: gemm_fmt<FMT_Q4_0>(c, s, x, T, kind, group, G, Y, max_items, st); break;
    case FMT_FP8_B128: gemm_fmt<FMT_FP8_B128>(c, s, x, T, kind, group, G, Y, max_items, st); break;
    case FMT_NVFP4: gemm_fmt<FMT_NVFP4>(c, s, x, T, kind, group, G, Y, max_items, st); break;
    default: break;
    }
}

void launch_combine(const CacheDev& c, const Scratch& s, float* out, int T, cudaStream_t st) {
    const size_t n = (size_t)T * c.H;
    const int blocks = (int)std::min<size_t>((n + 255) / 256, 4096);
    k_combine<<<blocks, 256, 0, st>>>(c, s, out, T);
}

}  // namespace moe
