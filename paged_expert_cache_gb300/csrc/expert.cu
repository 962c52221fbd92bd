// expert.cu -- the expert FFN of one layer call, read through the slot
// indirection, and the copy kernel that fills slots from the host store.
//
// Each CTA computes one 16-row tile of one matrix for one compute unit (a
// distinct expert of the call, or the shared expert) against up to eight of
// the unit's tokens at a time. Weights are dequantised in registers straight
// into m16n8k16 A fragments (see the slot layout in common.cuh); tokens are the
// B operand, staged in shared memory. The K dimension is split over the
// CTA's warps and the partial tiles are summed in a fixed warp order, so a
// token's result never depends on which slot its expert sits in, on whether
// the expert hit or missed, or on which other tokens shared the expert.
//
// Gate/up writes the SwiGLU activation a = silu(gate x) * (up x) per (token,
// pick) [Your GPU holds 24 GB... (cloudmash.blog), "The bus problem": gate,
// up and down projections]. Down writes one partial row block per (token,
// pick); the CTA that completes a row tile last sums the picks of every token
// in rank order with their router weights, plus the shared expert, into the
// output [same page, "The model that should not fit": routed plus shared].
#include "expert_dev.cuh"

namespace moe {

template <int FMT>
__global__ void __launch_bounds__(kGUWarps * 32, (FMT == FMT_Q4_0 || FMT == FMT_NVFP4) ? 3 : (FMT == FMT_FP8_B128 ? 2 : 1)) k_gateup(CacheDev c, Scratch s, const uint16_t* __restrict__ x,
                                                          int T, int kind, int group, int G) {
    extern __shared__ __align__(16) uint8_t smem[];
    griddep_wait();
    griddep_launch();
    UnitDesc d;
    const int u = fetch_unit(s, c.has_shared, kind, group, G, d);
    if (u < 0) return;
    note_miss_start(s, d);
    const int H = c.H, I = c.I, KC = H / 64, rt = blockIdx.x, k = c.k;
    const int ld = H + 8;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                      // [8][ld]
    float* red = reinterpret_cast<float*>(smem + (size_t)8 * ld * 2);      // [warps][2][128]
    const uint64_t mgu = matrix_stride(FMT, I, H);
    const uint8_t* Wg = reinterpret_cast<const uint8_t*>(d.src);
    const uint8_t* Wu = Wg + mgu;
    uint8_t* Dg = d.dst ? reinterpret_cast<uint8_t*>(d.dst) : nullptr;
    uint8_t* Du = Dg ? Dg + mgu : nullptr;
    if (Dg && rt == 0) {
        copy_matrix_tail<FMT>(Wg, Dg, I, H, threadIdx.x, blockDim.x);
        copy_matrix_tail<FMT>(Wu, Du, I, H, threadIdx.x, blockDim.x);
    }
    const int np = d.np;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cpw = (KC + kGUWarps - 1) / kGUWarps;
    for (int n0 = 0; n0 < np; n0 += 8) {
        uint8_t* dg = n0 == 0 ? Dg : nullptr;  // the slot is written on the first pass only
        uint8_t* du = n0 == 0 ? Du : nullptr;
        float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
        for (int c0 = 0; c0 < cpw; c0 += kMaxChunksInFlight) {
            Chunk<FMT> cg[kMaxChunksInFlight], cu[kMaxChunksInFlight];
#pragma unroll
            for (int i = 0; i < kMaxChunksInFlight; ++i) {
                const int kc = warp * cpw + c0 + i;
                if (c0 + i < cpw && kc < KC) {
                    load_chunk<FMT>(Wg, dg, I, H, rt, kc, lane, cg[i]);
                    load_chunk<FMT>(Wu, du, I, H, rt, kc, lane, cu[i]);
                }
            }
            if (c0 == 0) {
                // stage the tokens while the weight loads are in flight
                const int vpr = H / 8;
#pragma unroll 4
                for (int i = threadIdx.x; i < 8 * vpr; i += blockDim.x) {
                    const int nn = i / vpr, v = i - nn * vpr;
                    uint4 val = make_uint4(0u, 0u, 0u, 0u);
                    if (n0 + nn < np) {
                        const int t = pair_token(pair_at(s, d, n0 + nn), T, k);
                        val = *reinterpret_cast<const uint4*>(x + (size_t)t * H + v * 8);
                        if constexpr (FMT != FMT_BF16) {
                            // fp16 with the token's power-of-two prescale (exact)
                            const float sc = pow2f(-__ldg(s.tok_shift + t));
                            uint32_t w4[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float lo = __uint_as_float(w4[j] << 16) * sc;
                                const float hi = __uint_as_float(w4[j] & 0xffff0000u) * sc;
                                w4[j] = h2_as_u32(__floats2half2_rn(lo, hi));
                            }
                            val = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                    *reinterpret_cast<uint4*>(xs + (size_t)nn * ld + v * 8) = val;
                }
                __syncthreads();
            }
#pragma unroll
            for (int i = 0; i < kMaxChunksInFlight; ++i) {
                const int kc = warp * cpw + c0 + i;
                if (c0 + i < cpw && kc < KC) {
                    uint32_t b[1][4][2];
                    load_b(xs, ld, kc, lane, b[0]);
                    mma_chunk<FMT, 1>(cg[i], b, ag);
                    mma_chunk<FMT, 1>(cu[i], b, au);
                }
            }
        }
        const int g = lane >> 2, q = lane & 3;
        float* rg = red + (size_t)(warp * 2) * 128;
        float* ru = rg + 128;
        rg[g * 8 + 2 * q] = ag[0];
        rg[g * 8 + 2 * q + 1] = ag[1];
        rg[(g + 8) * 8 + 2 * q] = ag[2];
        rg[(g + 8) * 8 + 2 * q + 1] = ag[3];
        ru[g * 8 + 2 * q] = au[0];
        ru[g * 8 + 2 * q + 1] = au[1];
        ru[(g + 8) * 8 + 2 * q] = au[2];
        ru[(g + 8) * 8 + 2 * q + 1] = au[3];
        __syncthreads();
        if (threadIdx.x < 128) {
            const int row = threadIdx.x >> 3, col = threadIdx.x & 7;
            float gs = 0.f, us = 0.f;
#pragma unroll
            for (int w = 0; w < kGUWarps; ++w) {
                gs += red[(size_t)(w * 2) * 128 + threadIdx.x];
                us += red[(size_t)(w * 2 + 1) * 128 + threadIdx.x];
            }
            const int pair = n0 + col < np ? pair_at(s, d, n0 + col) : -1;
            float a = 0.f;
            if (pair >= 0) {
                const float up = FMT == FMT_BF16 ? 1.0f : pow2f(__ldg(s.tok_shift + pair_token(pair, T, k)));
                a = swiglu_scaled(gs, us, d.g[0], d.g[1], up);
            }
            store_act<FMT>(s, pair, I, rt * 16 + row, a);
        }
        __syncthreads();
    }
    if (Dg) {
        // this CTA's share of the missed record's down projection goes to the
        // slot now, so the whole record crosses the host link in one kernel
        // and the down kernel reads it from device memory
        const uint64_t mdn = matrix_stride(FMT, H, I);
        const uint64_t nvec = mdn / 16, per = (nvec + gridDim.x - 1) / gridDim.x;
        const uint64_t v0 = (uint64_t)rt * per, v1 = v0 + per < nvec ? v0 + per : nvec;
        const uint8_t* src = Wg + 2 * mgu;
        uint8_t* dst = Dg + 2 * mgu;
        constexpr int kBatch = 4;
        for (uint64_t v = v0 + threadIdx.x; v < v1; v += (uint64_t)blockDim.x * kBatch) {
            uint4 buf[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const uint64_t vi = v + (uint64_t)i * blockDim.x;
                if (vi < v1) buf[i] = ldg_stream(src + vi * 16);
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const uint64_t vi = v + (uint64_t)i * blockDim.x;
                if (vi < v1) stg_stream(dst + vi * 16, buf[i]);
            }
        }
    }
    note_miss_end(s, d);
}

template <int FMT>
__global__ void __launch_bounds__(kDNWarps * 32) k_down(CacheDev c, Scratch s, float* __restrict__ out, int T,
                                                        int kind, int group, int G, int bucket) {
    extern __shared__ __align__(16) uint8_t smem[];
    griddep_wait();
    griddep_launch();
    UnitDesc d;
    const int u = fetch_unit(s, c.has_shared, kind, group, G, d);
    if (u < 0) return;
    const int H = c.H, I = c.I, KC = I / 64, rt = blockIdx.x, k = c.k;
    const int ld = I + 8;
    uint16_t* xh = reinterpret_cast<uint16_t*>(smem);           // [8][ld] activations, high part
    uint16_t* xl = xh + (size_t)8 * ld;                          // [8][ld] low part
    float* red = reinterpret_cast<float*>(xl + (size_t)8 * ld);  // [warps][128]
    const uint64_t mgu = matrix_stride(FMT, I, H);
    // a missed expert was written to its slot by the gate/up kernel
    const uint8_t* Wd = reinterpret_cast<const uint8_t*>(d.dst ? d.dst : d.src) + 2 * mgu;
    const int np = d.np;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cpw = (KC + kDNWarps - 1) / kDNWarps;
    __shared__ int psh[8];  // the prescale of each of the eight pairs' activations
    for (int n0 = 0; n0 < np; n0 += 8) {
        if (threadIdx.x < 8)
            psh[threadIdx.x] = n0 + (int)threadIdx.x < np ? pair_act_shift<FMT>(s, pair_at(s, d, n0 + threadIdx.x)) : 0;
        __syncthreads();
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int c0 = 0; c0 < cpw; c0 += kMaxChunksInFlight) {
            Chunk<FMT> cd[kMaxChunksInFlight];
#pragma unroll
            for (int i = 0; i < kMaxChunksInFlight; ++i) {
                const int kc = warp * cpw + c0 + i;
                if (c0 + i < cpw && kc < KC) load_chunk<FMT>(Wd, nullptr, H, I, rt, kc, lane, cd[i]);
            }
            if (c0 == 0) {
                // split each fp32 activation into two 16-bit parts, hi + lo;
                // all of a thread's loads are issued before any is used
                const int vpr = I / 4;
                constexpr int kStage = 12;
                float4 av4[kStage];
#pragma unroll
                for (int r = 0; r < kStage; ++r) {
                    const int i = threadIdx.x + r * blockDim.x;
                    const int nn = i / vpr, v = i - nn * vpr;
                    av4[r] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (i < 8 * vpr && n0 + nn < np)
                        av4[r] = *reinterpret_cast<const float4*>(s.act + (size_t)pair_at(s, d, n0 + nn) * I + v * 4);
                }
                for (int r = 0; r * (int)blockDim.x < 8 * vpr; ++r) {
                    const int i = threadIdx.x + r * blockDim.x;
                    if (i >= 8 * vpr) break;
                    const int nn = i / vpr, v = i - nn * vpr;
                    float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (r < kStage) {
#pragma unroll
                        for (int q = 0; q < kStage; ++q)
                            if (q == r) a4 = av4[q];
                    } else if (n0 + nn < np) {
                        a4 = *reinterpret_cast<const float4*>(s.act + (size_t)pair_at(s, d, n0 + nn) * I + v * 4);
                    }
                    const float sc = pow2f(-psh[nn]);
                    const float av[4] = {a4.x * sc, a4.y * sc, a4.z * sc, a4.w * sc};
                    uint16_t hv[4], lv[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) split_hi_lo<FMT>(av[j], hv[j], lv[j]);
                    *reinterpret_cast<uint2*>(xh + (size_t)nn * ld + v * 4) =
                        make_uint2(hv[0] | ((uint32_t)hv[1] << 16), hv[2] | ((uint32_t)hv[3] << 16));
                    *reinterpret_cast<uint2*>(xl + (size_t)nn * ld + v * 4) =
                        make_uint2(lv[0] | ((uint32_t)lv[1] << 16), lv[2] | ((uint32_t)lv[3] << 16));
                }
                __syncthreads();
            }
#pragma unroll
            for (int i = 0; i < kMaxChunksInFlight; ++i) {
                const int kc = warp * cpw + c0 + i;
                if (c0 + i < cpw && kc < KC) {
                    uint32_t b[2][4][2];
                    load_b(xh, ld, kc, lane, b[0]);
                    load_b(xl, ld, kc, lane, b[1]);
                    mma_chunk<FMT, 2>(cd[i], b, acc);
                }
            }
        }
        const int g = lane >> 2, q = lane & 3;
        float* rw = red + (size_t)warp * 128;
        rw[g * 8 + 2 * q] = acc[0];
        rw[g * 8 + 2 * q + 1] = acc[1];
        rw[(g + 8) * 8 + 2 * q] = acc[2];
        rw[(g + 8) * 8 + 2 * q + 1] = acc[3];
        __syncthreads();
        {
            const int row = threadIdx.x >> 3, col = threadIdx.x & 7;  // 128 threads = 16 x 8
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kDNWarps; ++w) sum += red[(size_t)w * 128 + threadIdx.x];
            if (n0 + col < np) {
                const int pair = pair_at(s, d, n0 + col);
                s.part[(size_t)pair * H + rt * 16 + row] = sum * d.g[2] * pow2f(psh[col]);
            }
        }
        __syncthreads();
    }
    // the CTA that finishes this row tile last combines it for every token
    __threadfence();
    __syncthreads();
    __shared__ int last;
    if (threadIdx.x == 0) last = atomicAdd(s.tile_done + rt, 1u) == (unsigned)(s.plan->n_units - 1);
    __syncthreads();
    if (!last) return;
    __threadfence();
    for (int i = threadIdx.x; i < T * 16; i += blockDim.x) {
        const int t = i >> 4, row = i & 15;
        const size_t col = (size_t)rt * 16 + row;
        float y = 0.f;
        for (int j = 0; j < k; ++j) y = fmaf(s.wts[t * k + j], __ldcg(s.part + (size_t)(t * k + j) * H + col), y);
        if (c.has_shared) y += __ldcg(s.part + (size_t)(T * k + t) * H + col);
        out[(size_t)t * H + col] = y;
    }
    if (threadIdx.x == 0) {
        s.tile_done[rt] = 0u;
        // the last row tile of the call books the time misses were streamed
        if (atomicAdd(s.tiles_done, 1u) == gridDim.x - 1) {
            __threadfence();
            const unsigned long long t1 = atomicAdd(s.copy_t1, 0ull);
            if (t1) {
                const unsigned long long t0 = atomicAdd(s.copy_t0, 0ull);
                c.stats[bucket * 5 + 4] += t1 - t0;
                *s.copy_t0 = ~0ull;
                *s.copy_t1 = 0ull;
            }
            *s.tiles_done = 0u;
        }
    }
}

// Down projection of a decode call, one CTA per 16-row output tile over every
// unit of the call (down_rows_tile); the descriptors and activations are
// staged in shared memory first.
template <int FMT>
__global__ void __launch_bounds__(kDRWarps * 32, 1) k_down_rows(CacheDev c, Scratch s, float* __restrict__ out,
                                                                 int T, int U, int bucket) {
    extern __shared__ __align__(16) uint8_t smem[];
    griddep_wait();
    griddep_launch();
    const int I = c.I;
    const int n_units = s.plan->n_units;
    const int P = T * c.k + (c.has_shared ? T : 0);
    const int ld = I + 8;
    UnitDesc* sd = reinterpret_cast<UnitDesc*>(smem);
    uint16_t* ah = reinterpret_cast<uint16_t*>(smem + (size_t)U * sizeof(UnitDesc));
    uint16_t* al = ah + (size_t)(P + 1) * ld;
    float* ps = reinterpret_cast<float*>(al + (size_t)(P + 1) * ld);
    const int tid = threadIdx.x, nthr = blockDim.x;
    {
        const int nw = n_units * (int)(sizeof(UnitDesc) / 16);
        const uint4* src = reinterpret_cast<const uint4*>(s.units);
        uint4* dst = reinterpret_cast<uint4*>(sd);
        for (int j = tid; j < nw; j += nthr) dst[j] = __ldcg(src + j);
    }
    __shared__ int psh[kDecodeMaxTokens * (kMaxTopK + 1)];  // the pairs' activation prescales
    down_stage_act<FMT>(s, P, I, ah, al, psh);
    __syncthreads();
    down_rows_tile<FMT>(c, s, sd, n_units, T, blockIdx.x, ah, al, psh, ps, s.wts, out);
    if (tid == 0 && atomicAdd(s.tiles_done, 1u) == gridDim.x - 1) {
        // the last tile of the call books the time misses were streamed
        __threadfence();
        const unsigned long long t1 = atomicAdd(s.copy_t1, 0ull);
        if (t1) {
            const unsigned long long t0 = atomicAdd(s.copy_t0, 0ull);
            c.stats[bucket * 5 + 4] += t1 - t0;
            *s.copy_t0 = ~0ull;
            *s.copy_t1 = 0ull;
        }
        *s.tiles_done = 0u;
    }
}

// ---------------------------------------------------------------------------
// Record copies host store -> slots (or the prefill arena), pulled by the GPU
// from the mapped pinned store: entries [first, first + count) of the copy
// list, bounded by the plan's n_fill.
// ---------------------------------------------------------------------------
constexpr int kCopyThreads = 256;
constexpr uint64_t kCopyChunk = 32768;

__global__ void __launch_bounds__(kCopyThreads) k_copy(CacheDev c, Scratch s, int first, int count, int bucket) {
    griddep_wait();
    const int n = min(s.plan->n_fill - first, count);
    if (n <= 0) return;
    if (threadIdx.x == 0) atomicMin(s.copy_t0, globaltimer_ns());
    const uint64_t bytes = c.slot_bytes;
    const int cpr = (int)((bytes + kCopyChunk - 1) / kCopyChunk);
    const long long total = (long long)n * cpr;
    for (long long w = blockIdx.x; w < total; w += gridDim.x) {
        const int r = first + (int)(w / cpr), ch = (int)(w % cpr);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(s.copy_src[r]) + (size_t)ch * kCopyChunk;
        uint8_t* dst = reinterpret_cast<uint8_t*>(s.copy_dst[r]) + (size_t)ch * kCopyChunk;
        const uint64_t rem = bytes - (uint64_t)ch * kCopyChunk;
        const int nv = (int)((rem < kCopyChunk ? rem : kCopyChunk) / 16);
        for (int v0 = threadIdx.x; v0 < nv; v0 += kCopyThreads * 8) {
            uint4 buf[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int v = v0 + i * kCopyThreads;
                if (v < nv) buf[i] = ldg_stream(src + (size_t)v * 16);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int v = v0 + i * kCopyThreads;
                if (v < nv) *reinterpret_cast<uint4*>(dst + (size_t)v * 16) = buf[i];
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicMax(s.copy_t1, globaltimer_ns());
        const unsigned ticket = atomicAdd(s.copy_done, 1u);
        if (ticket == gridDim.x - 1) {
            __threadfence();
            const unsigned long long t0 = atomicAdd(s.copy_t0, 0ull), t1 = atomicAdd(s.copy_t1, 0ull);
            c.stats[bucket * 5 + 4] += t1 - t0;
            *s.copy_t0 = ~0ull;
            *s.copy_t1 = 0ull;
            *s.copy_done = 0u;
        }
    }
}

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------
static int g_copy_ctas = 0;

void launch_copy(const CacheDev& c, const Scratch& s, int first, int count, int bucket, cudaStream_t st,
                 bool beside_compute) {
    if (!g_copy_ctas) {
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_copy_ctas = sms > 0 ? sms : 148;
    }
    // alone: two CTAs per SM; beside the GEMMs of another group: a quarter of
    // the SMs, whose loads in flight (~1 MB) still cover the host link
    const int ctas = beside_compute ? (g_copy_ctas + 3) / 4 : 2 * g_copy_ctas;
    k_copy<<<ctas, kCopyThreads, 0, st>>>(c, s, first, count, bucket);
}

template <int FMT>
static void gateup_fmt(const CacheDev& c, const Scratch& s, const uint16_t* x, int T, int kind, int group, int G,
                       int units, cudaStream_t st, bool pdl) {
    const size_t sm = (size_t)8 * (c.H + 8) * 2 + (size_t)kGUWarps * 2 * 128 * 4;
    static size_t set = 0;
    if (sm > set) {
        cudaFuncSetAttribute(k_gateup<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        set = sm;
    }
    dim3 grid(c.I / 16, units);
    launch_ex(k_gateup<FMT>, grid, dim3(kGUWarps * 32), sm, st, pdl, c, s, x, T, kind, group, G);
}

template <int FMT>
static void down_fmt(const CacheDev& c, const Scratch& s, float* out, int T, int kind, int group, int G, int units,
                     int bucket, cudaStream_t st, bool pdl) {
    const size_t sm = (size_t)2 * 8 * (c.I + 8) * 2 + (size_t)kDNWarps * 128 * 4;
    static size_t set = 0;
    if (sm > set) {
        cudaFuncSetAttribute(k_down<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        set = sm;
    }
    dim3 grid(c.H / 16, units);
    launch_ex(k_down<FMT>, grid, dim3(kDNWarps * 32), sm, st, pdl, c, s, out, T, kind, group, G, bucket);
}

template <int FMT>
static bool down_rows_fmt(const CacheDev& c, const Scratch& s, float* out, int T, int units, int bucket,
                          cudaStream_t st, bool pdl) {
    const int P = T * c.k + (c.has_shared ? T : 0);
    const size_t sm = down_rows_smem(c.I, c.I / 64, units, P);
    if (sm > 200 * 1024) return false;
    static size_t set = 0;
    if (sm > set) {
        cudaFuncSetAttribute(k_down_rows<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        set = 200 * 1024;
    }
    launch_ex(k_down_rows<FMT>, dim3(c.H / 16), dim3(kDRWarps * 32), sm, st, pdl, c, s, out, T, units, bucket);
    return true;
}

// Decode down projection: the row-tile kernel when its staging fits in
// shared memory, else the per-unit kernel with a global combine.
bool launch_down_rows(const CacheDev& c, const Scratch& s, float* out, int T, int units, int bucket, cudaStream_t st,
                      bool pdl) {
    switch (c.fmt) {
    case FMT_BF16: return down_rows_fmt<FMT_BF16>(c, s, out, T, units, bucket, st, pdl);
    case FMT_Q4_0: return down_rows_fmt<FMT_Q4_0>(c, s, out, T, units, bucket, st, pdl);
    case FMT_FP8_B128: return down_rows_fmt<FMT_FP8_B128>(c, s, out, T, units, bucket, st, pdl);
    case FMT_NVFP4: return down_rows_fmt<FMT_NVFP4>(c, s, out, T, units, bucket, st, pdl);
    }
    return false;
}

void launch_gateup(const CacheDev& c, const Scratch& s, const uint16_t* x, int T, int kind, int group, int G,
                   int units, cudaStream_t st, bool pdl) {
    switch (c.fmt) {
    case FMT_BF16: gateup_fmt<FMT_BF16>(c, s, x, T, kind, group, G, units, st, pdl); break;
    case FMT_Q4_0: gateup_fmt<FMT_Q4_0>(c, s, x, T, kind, group, G, units, st, pdl); break;
    case FMT_FP8_B128: gateup_fmt<FMT_FP8_B128>(c, s, x, T, kind, group, G, units, st, pdl); break;
    case FMT_NVFP4: gateup_fmt<FMT_NVFP4>(c, s, x, T, kind, group, G, units, st, pdl); break;
    }
}

void launch_down(const CacheDev& c, const Scratch& s, float* out, int T, int kind, int group, int G, int units,
                 int bucket, cudaStream_t st, bool pdl) {
    switch (c.fmt) {
    case FMT_BF16: down_fmt<FMT_BF16>(c, s, out, T, kind, group, G, units, bucket, st, pdl); break;
    case FMT_Q4_0: down_fmt<FMT_Q4_0>(c, s, out, T, kind, group, G, units, bucket, st, pdl); break;
    case FMT_FP8_B128: down_fmt<FMT_FP8_B128>(c, s, out, T, kind, group, G, units, bucket, st, pdl); break;
    case FMT_NVFP4: down_fmt<FMT_NVFP4>(c, s, out, T, kind, group, G, units, bucket, st, pdl); break;
    }
}

}  // namespace moe
