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
#include "common.cuh"

namespace moe {

template <int FMT> struct Chunk;
template <> struct Chunk<FMT_Q4_0> { uint4 q; uint2 sc; };
template <> struct Chunk<FMT_NVFP4> { uint4 q; uint2 sc; };
template <> struct Chunk<FMT_FP8_B128> { uint4 q0, q1; float sc; };
template <> struct Chunk<FMT_BF16> { uint4 q[4]; };

// Loads the lane's share of chunk (rt, kc) of a matrix M (R rows, C cols).
// When D is not null (a missed expert read from the host store), the same
// bytes are written to the slot D at the same offsets, so the slot ends up
// holding the record without a separate copy pass.
template <int FMT>
__device__ __forceinline__ void load_chunk(const uint8_t* M, uint8_t* D, int R, int C, int rt, int kc, int lane,
                                           Chunk<FMT>& ch) {
    const int KC = C / 64;
    const size_t tile = (size_t)rt * KC + kc;
    if constexpr (FMT == FMT_Q4_0 || FMT == FMT_NVFP4) {
        const size_t qo = (tile * 32 + lane) * 16;
        const size_t so = (size_t)R * C / 2 + (tile * 8 + (lane >> 2)) * 8;
        ch.q = ldg_stream(M + qo);
        if (D) {
            ch.sc = ldg_stream8(M + so);
            stg_stream(D + qo, ch.q);
            if ((lane & 3) == 0) stg_stream8(D + so, ch.sc);
        } else {
            ch.sc = __ldg(reinterpret_cast<const uint2*>(M + so));
        }
    } else if constexpr (FMT == FMT_FP8_B128) {
        const size_t qo = (tile * 32 + lane) * 32;
        ch.q0 = ldg_stream(M + qo);
        ch.q1 = ldg_stream(M + qo + 16);
        const int nct = (C + 127) / 128;
        ch.sc = __ldg(reinterpret_cast<const float*>(M + (size_t)R * C) + (size_t)((rt * 16) / 128) * nct + (kc * 64) / 128);
        if (D) {
            stg_stream(D + qo, ch.q0);
            stg_stream(D + qo + 16, ch.q1);
        }
    } else {
        const size_t qo = (tile * 32 + lane) * 64;
#pragma unroll
        for (int i = 0; i < 4; ++i) ch.q[i] = ldg_stream(M + qo + 16 * i);
        if (D) {
#pragma unroll
            for (int i = 0; i < 4; ++i) stg_stream(D + qo + 16 * i, ch.q[i]);
        }
    }
}

// The bytes of a matrix that no lane's chunk covers (block-FP8 tile scales and
// the padding up to the 16-byte matrix stride), copied by one CTA per matrix.
template <int FMT>
__device__ __forceinline__ void copy_matrix_tail(const uint8_t* M, uint8_t* D, int R, int C) {
    const size_t begin = FMT == FMT_FP8_B128 ? (size_t)R * C : matrix_bytes(FMT, R, C);
    const size_t end = matrix_stride(FMT, R, C);
    for (size_t i = begin + threadIdx.x * 4; i < end; i += blockDim.x * 4)
        *reinterpret_cast<uint32_t*>(D + i) = *reinterpret_cast<const uint32_t*>(M + i);
}

// acc += A(chunk) * B over the chunk's four k16 steps, for NB B operands
// (NB = 2: the same weights against a hi and a lo part of the activations).
template <int FMT, int NB>
__device__ __forceinline__ void mma_chunk(const Chunk<FMT>& ch, const uint32_t (&b)[NB][4][2], float acc[4]) {
    if constexpr (FMT == FMT_Q4_0) {
        const uint32_t w[4] = {ch.q.x, ch.q.y, ch.q.z, ch.q.w};
        const float d[4] = {__low2float(u32_as_h2(ch.sc.x)), __high2float(u32_as_h2(ch.sc.x)),
                            __low2float(u32_as_h2(ch.sc.y)), __high2float(u32_as_h2(ch.sc.y))};
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
            float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ss = 0; ss < 2; ++ss) {
                const int s = blk * 2 + ss;
                uint32_t a[4];
                q4_to_frag(w[s], a);
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) mma_f16(t, a, b[nb][s][0], b[nb][s][1]);
            }
            const float dr0 = d[blk], dr8 = d[2 + blk];  // rows g and g+8 of this 32-column block
            acc[0] = fmaf(dr0, t[0], acc[0]);
            acc[1] = fmaf(dr0, t[1], acc[1]);
            acc[2] = fmaf(dr8, t[2], acc[2]);
            acc[3] = fmaf(dr8, t[3], acc[3]);
        }
    } else if constexpr (FMT == FMT_NVFP4) {
        const uint32_t w[4] = {ch.q.x, ch.q.y, ch.q.z, ch.q.w};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint32_t scw = s < 2 ? ch.sc.x : ch.sc.y;
            const __half2 sh = u32_as_h2(e4m3x2_to_h2((scw >> (16 * (s & 1))) & 0xffffu));
            const __half2 sg = __low2half2(sh), s8 = __high2half2(sh);
            uint32_t a[4];
            a[0] = h2_as_u32(__hmul2(u32_as_h2(e2m1x2_to_h2(w[s] & 0xffu)), sg));
            a[1] = h2_as_u32(__hmul2(u32_as_h2(e2m1x2_to_h2((w[s] >> 8) & 0xffu)), s8));
            a[2] = h2_as_u32(__hmul2(u32_as_h2(e2m1x2_to_h2((w[s] >> 16) & 0xffu)), sg));
            a[3] = h2_as_u32(__hmul2(u32_as_h2(e2m1x2_to_h2(w[s] >> 24)), s8));
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_f16(acc, a, b[nb][s][0], b[nb][s][1]);
        }
    } else if constexpr (FMT == FMT_FP8_B128) {
        const uint32_t w[8] = {ch.q0.x, ch.q0.y, ch.q0.z, ch.q0.w, ch.q1.x, ch.q1.y, ch.q1.z, ch.q1.w};
        float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            uint32_t a[4];
            a[0] = e4m3x2_to_h2(w[2 * s] & 0xffffu);
            a[1] = e4m3x2_to_h2(w[2 * s] >> 16);
            a[2] = e4m3x2_to_h2(w[2 * s + 1] & 0xffffu);
            a[3] = e4m3x2_to_h2(w[2 * s + 1] >> 16);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_f16(t, a, b[nb][s][0], b[nb][s][1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = fmaf(ch.sc, t[i], acc[i]);
    } else {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint32_t a[4] = {ch.q[s].x, ch.q[s].y, ch.q[s].z, ch.q[s].w};
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_bf16(acc, a, b[nb][s][0], b[nb][s][1]);
        }
    }
}

// B fragments of the four k-steps of chunk kc from a [8][ld] 16-bit tile.
__device__ __forceinline__ void load_b(const uint16_t* xs, int ld, int kc, int lane, uint32_t (&b)[4][2]) {
    const uint16_t* row = xs + (size_t)(lane & 7) * ld + kc * 64 + (lane >> 3) * 8;
    ldmatrix_x4(b[0][0], b[0][1], b[1][0], b[1][1], row);
    ldmatrix_x4(b[2][0], b[2][1], b[3][0], b[3][1], row + 32);
}

// Compute unit of blockIdx.y for a launch over unit range `kind`:
// 0 = every unit of a decode call; 1 = prefill experts read in place, plus
// the shared expert; 2 = prefill staging group `group`.
__device__ __forceinline__ int map_unit(const Plan* p, int has_shared, int kind, int group, int G, int y) {
    if (kind == 0) return y < p->n_units ? y : -1;
    if (kind == 1) {
        if (y < p->n_hit) return y;
        if (has_shared && y == p->n_hit) return p->n_uniq;
        return -1;
    }
    if (y >= G) return -1;
    int u = p->n_hit + group * G + y;
    return u < p->n_uniq ? u : -1;
}

// The unit of this CTA and its descriptor. For a decode launch (kind 0) the
// unit index is the CTA's y coordinate, so the descriptor load is issued
// together with the plan load instead of after it.
__device__ __forceinline__ int fetch_unit(const Scratch& s, int has_shared, int kind, int group, int G,
                                          UnitDesc& d) {
    if (kind == 0) {
        const int y = blockIdx.y;
        const int n_units = s.plan->n_units;
        d = s.units[y];
        return y < n_units ? y : -1;
    }
    const int u = map_unit(s.plan, has_shared, kind, group, G, blockIdx.y);
    if (u >= 0) d = s.units[u];
    return u;
}

__device__ __forceinline__ int pair_at(const Scratch& s, const UnitDesc& d, int i) {
    if (i >= 8) return s.unit_pairs[d.pstart + i];
    int r = d.pair8[0];
#pragma unroll
    for (int j = 1; j < 8; ++j)
        if (i == j) r = d.pair8[j];  // constant indices keep the descriptor in registers
    return r;
}

__device__ __forceinline__ int pair_token(int pair, int T, int k) { return pair < T * k ? pair / k : pair - T * k; }

constexpr int kGUWarps = 8;
constexpr int kDNWarps = 4;
constexpr int kMaxChunksInFlight = 4;

__device__ __forceinline__ void note_miss_start(const Scratch& s, const UnitDesc& d) {
    if (d.dst && threadIdx.x == 0) atomicMin(s.copy_t0, globaltimer_ns());
}
__device__ __forceinline__ void note_miss_end(const Scratch& s, const UnitDesc& d) {
    if (d.dst && threadIdx.x == 0) atomicMax(s.copy_t1, globaltimer_ns());
}

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
        copy_matrix_tail<FMT>(Wg, Dg, I, H);
        copy_matrix_tail<FMT>(Wu, Du, I, H);
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
                            uint32_t w4[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float lo = __uint_as_float(w4[j] << 16);
                                const float hi = __uint_as_float(w4[j] & 0xffff0000u);
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
            if (n0 + col < np) {
                const int pair = pair_at(s, d, n0 + col);
                s.act[(size_t)pair * I + rt * 16 + row] = silu_f(gs * d.g[0]) * (us * d.g[1]);
            }
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
    for (int n0 = 0; n0 < np; n0 += 8) {
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
                    const float av[4] = {a4.x, a4.y, a4.z, a4.w};
                    uint16_t hv[4], lv[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if constexpr (FMT == FMT_BF16) {
                            __nv_bfloat16 h = __float2bfloat16_rn(av[j]);
                            __nv_bfloat16 l = __float2bfloat16_rn(av[j] - __bfloat162float(h));
                            hv[j] = *reinterpret_cast<uint16_t*>(&h);
                            lv[j] = *reinterpret_cast<uint16_t*>(&l);
                        } else {
                            __half h = __float2half_rn(av[j]);
                            __half l = __float2half_rn(av[j] - __half2float(h));
                            hv[j] = *reinterpret_cast<uint16_t*>(&h);
                            lv[j] = *reinterpret_cast<uint16_t*>(&l);
                        }
                    }
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
                s.part[(size_t)pair * H + rt * 16 + row] = sum * d.g[2];
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

// ---------------------------------------------------------------------------
// Down projection of a decode call, one CTA per 16-row tile of the output
// over every unit of the call. The unit descriptors and every pair's
// activation (split into hi + lo 16-bit parts) are staged in shared memory
// once; warps take (unit, group of kDRChunks chunks) items with all their
// weight loads in flight; each item's partial tile goes to shared memory per
// (chunk group, pair, row), and the CTA sums the groups in order, weights the
// picks in rank order and adds the shared expert. No partial leaves the SM.
// ---------------------------------------------------------------------------
constexpr int kDRWarps = 16;
constexpr int kDRChunks = 4;

__host__ __device__ inline size_t down_rows_smem(int I, int KC, int U, int P) {
    const size_t ld = (size_t)I + 8;
    const int ncg = (KC + kDRChunks - 1) / kDRChunks;
    return (size_t)U * sizeof(UnitDesc) + 2 * (size_t)(P + 1) * ld * 2 + (size_t)ncg * P * 16 * 4;
}

template <int FMT>
__global__ void __launch_bounds__(kDRWarps * 32, 1) k_down_rows(CacheDev c, Scratch s, float* __restrict__ out,
                                                                 int T, int U, int bucket) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int IB = FMT == FMT_BF16 ? 1 : 2;  // items a warp keeps in flight
    griddep_wait();
    griddep_launch();
    const int H = c.H, I = c.I, KC = I / 64, rt = blockIdx.x, k = c.k;
    const int n_units = s.plan->n_units;
    const int P = T * k + (c.has_shared ? T : 0);
    const int ld = I + 8;
    const int ncg = (KC + kDRChunks - 1) / kDRChunks;
    UnitDesc* sd = reinterpret_cast<UnitDesc*>(smem);
    uint16_t* ah = reinterpret_cast<uint16_t*>(smem + (size_t)U * sizeof(UnitDesc));
    uint16_t* al = ah + (size_t)(P + 1) * ld;
    float* ps = reinterpret_cast<float*>(al + (size_t)(P + 1) * ld);
    const int tid = threadIdx.x, nthr = blockDim.x;
    // stage the descriptors (uint4 words) and the activations (float4 -> hi/lo)
    {
        const int nw = n_units * (int)(sizeof(UnitDesc) / 16);
        const uint4* src = reinterpret_cast<const uint4*>(s.units);
        uint4* dst = reinterpret_cast<uint4*>(sd);
        const int vpr = I / 4;
        const int nv = P * vpr;
        constexpr int B = 4;
        for (int base = tid; base < nw + nv; base += nthr * B) {
            float4 v[B];
            uint4 w[B];
#pragma unroll
            for (int i = 0; i < B; ++i) {
                const int j = base + i * nthr;
                if (j < nw) w[i] = __ldcg(src + j);
                else if (j < nw + nv) v[i] = __ldcg(reinterpret_cast<const float4*>(s.act) + (j - nw));
            }
#pragma unroll
            for (int i = 0; i < B; ++i) {
                const int j = base + i * nthr;
                if (j < nw) {
                    dst[j] = w[i];
                } else if (j < nw + nv) {
                    const int pr = (j - nw) / vpr, cv = (j - nw) - pr * vpr;
                    const float av[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                    uint16_t hv[4], lv[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if constexpr (FMT == FMT_BF16) {
                            __nv_bfloat16 h = __float2bfloat16_rn(av[q]);
                            __nv_bfloat16 l = __float2bfloat16_rn(av[q] - __bfloat162float(h));
                            hv[q] = *reinterpret_cast<uint16_t*>(&h);
                            lv[q] = *reinterpret_cast<uint16_t*>(&l);
                        } else {
                            __half h = __float2half_rn(av[q]);
                            __half l = __float2half_rn(av[q] - __half2float(h));
                            hv[q] = *reinterpret_cast<uint16_t*>(&h);
                            lv[q] = *reinterpret_cast<uint16_t*>(&l);
                        }
                    }
                    *reinterpret_cast<uint2*>(ah + (size_t)pr * ld + cv * 4) =
                        make_uint2(hv[0] | ((uint32_t)hv[1] << 16), hv[2] | ((uint32_t)hv[3] << 16));
                    *reinterpret_cast<uint2*>(al + (size_t)pr * ld + cv * 4) =
                        make_uint2(lv[0] | ((uint32_t)lv[1] << 16), lv[2] | ((uint32_t)lv[3] << 16));
                }
            }
        }
        for (int i = tid; i < ld / 2; i += nthr) {  // the zero row used for padding columns
            reinterpret_cast<uint32_t*>(ah + (size_t)P * ld)[i] = 0u;
            reinterpret_cast<uint32_t*>(al + (size_t)P * ld)[i] = 0u;
        }
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
    const int n_items = n_units * ncg;
    for (int it0 = warp * IB; it0 < n_items; it0 += kDRWarps * IB) {
        Chunk<FMT> ch[IB][kDRChunks];
#pragma unroll
        for (int b = 0; b < IB; ++b) {
            const int it = it0 + b;
            if (it >= n_items) break;
            const UnitDesc& d = sd[it / ncg];
            const int cg = it - (it / ncg) * ncg;
            const uint8_t* W = reinterpret_cast<const uint8_t*>(d.dst ? d.dst : d.src) + 2 * matrix_stride(FMT, I, H);
#pragma unroll
            for (int i = 0; i < kDRChunks; ++i) {
                const int kc = cg * kDRChunks + i;
                if (kc < KC) load_chunk<FMT>(W, nullptr, H, I, rt, kc, lane, ch[b][i]);
            }
        }
#pragma unroll
        for (int b = 0; b < IB; ++b) {
            const int it = it0 + b;
            if (it >= n_items) break;
            const UnitDesc& d = sd[it / ncg];
            const int cg = it - (it / ncg) * ncg;
            for (int n0 = 0; n0 < d.np; n0 += 8) {
                // this lane's ldmatrix row: token column (lane & 7) of the tile
                const int col = lane & 7;
                const int pr = n0 + col < d.np ? (n0 + col < 8 ? d.pair8[n0 + col] : s.unit_pairs[d.pstart + n0 + col]) : P;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < kDRChunks; ++i) {
                    const int kc = cg * kDRChunks + i;
                    if (kc >= KC) break;
                    if (n0 > 0) load_chunk<FMT>(reinterpret_cast<const uint8_t*>(d.dst ? d.dst : d.src) +
                                                    2 * matrix_stride(FMT, I, H), nullptr, H, I, rt, kc, lane, ch[b][i]);
                    uint32_t bf[2][4][2];
                    const uint16_t* rh = ah + (size_t)pr * ld + kc * 64 + (lane >> 3) * 8;
                    const uint16_t* rl = al + (size_t)pr * ld + kc * 64 + (lane >> 3) * 8;
                    ldmatrix_x4(bf[0][0][0], bf[0][0][1], bf[0][1][0], bf[0][1][1], rh);
                    ldmatrix_x4(bf[0][2][0], bf[0][2][1], bf[0][3][0], bf[0][3][1], rh + 32);
                    ldmatrix_x4(bf[1][0][0], bf[1][0][1], bf[1][1][0], bf[1][1][1], rl);
                    ldmatrix_x4(bf[1][2][0], bf[1][2][1], bf[1][3][0], bf[1][3][1], rl + 32);
                    mma_chunk<FMT, 2>(ch[b][i], bf, acc);
                }
                const float gd = d.g[2];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int cc = 2 * q + c2;
                        if (n0 + cc < d.np) {
                            const int pair = n0 + cc < 8 ? d.pair8[n0 + cc] : s.unit_pairs[d.pstart + n0 + cc];
                            ps[((size_t)cg * P + pair) * 16 + g + 8 * h2] = acc[2 * h2 + c2] * gd;
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < T * 16; i += nthr) {
        const int t = i >> 4, row = i & 15;
        float y = 0.f;
        for (int j = 0; j < k; ++j) {
            const int pair = t * k + j;
            float v = 0.f;
            for (int cg = 0; cg < ncg; ++cg) v += ps[((size_t)cg * P + pair) * 16 + row];
            y = fmaf(s.wts[pair], v, y);
        }
        if (c.has_shared) {
            const int pair = T * k + t;
            float v = 0.f;
            for (int cg = 0; cg < ncg; ++cg) v += ps[((size_t)cg * P + pair) * 16 + row];
            y += v;
        }
        out[(size_t)t * H + (size_t)rt * 16 + row] = y;
    }
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

void launch_copy(const CacheDev& c, const Scratch& s, int first, int count, int bucket, cudaStream_t st) {
    if (!g_copy_ctas) {
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_copy_ctas = 2 * (sms > 0 ? sms : 148);
    }
    k_copy<<<g_copy_ctas, kCopyThreads, 0, st>>>(c, s, first, count, bucket);
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
