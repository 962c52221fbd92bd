// expert_dev.cuh -- device routines of the expert FFN (dequantising loads,
// tensor-core chunks, the row-tile down projection), shared by the expert
// kernels (expert.cu) and the fused decode-layer kernel (layer.cu).
//
// Gate/up computes the SwiGLU activation a = silu(gate x) * (up x) per
// (token, pick) [Your GPU holds 24 GB... (cloudmash.blog), "The bus problem":
// gate, up and down projections]; down sums the picks of every token in rank
// order with their router weights, plus the shared expert [same page, "The
// model that should not fit": routed plus shared].
#pragma once

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

// Asks L2 for row tiles rt0 .. rt0 + nrt - 1 of a slot matrix (R rows, C
// columns) whole: their codes are one contiguous range and so are their
// scales (block-FP8: the 128-row blocks of scales they use). Thread `part` of
// nparts issues its share of 16 KB pieces.
template <int FMT>
__device__ __forceinline__ void prefetch_rows(const uint8_t* M, int R, int C, int rt0, int nrt, int part, int nparts) {
    const int KC = C / 64;
    uint64_t off[2], len[2];
    int nr = 1;
    if constexpr (FMT == FMT_Q4_0 || FMT == FMT_NVFP4) {
        off[0] = (uint64_t)rt0 * KC * 512;
        len[0] = (uint64_t)nrt * KC * 512;
        off[1] = (uint64_t)R * C / 2 + (uint64_t)rt0 * KC * 64;
        len[1] = (uint64_t)nrt * KC * 64;
        nr = 2;
    } else if constexpr (FMT == FMT_FP8_B128) {
        const int nct = (C + 127) / 128;
        off[0] = (uint64_t)rt0 * KC * 1024;
        len[0] = (uint64_t)nrt * KC * 1024;
        const uint64_t s0 = (uint64_t)R * C + (uint64_t)((rt0 * 16) / 128) * nct * 4;
        const uint64_t s1 = (uint64_t)R * C + (uint64_t)((rt0 * 16 + nrt * 16 + 127) / 128) * nct * 4;
        off[1] = s0 & ~15ull;
        len[1] = ((s1 + 15) & ~15ull) - off[1];
        nr = 2;
    } else {
        off[0] = (uint64_t)rt0 * KC * 2048;
        len[0] = (uint64_t)nrt * KC * 2048;
    }
    constexpr uint64_t kPiece = 16384;
    int idx = 0;
    for (int r = 0; r < nr; ++r)
        for (uint64_t o = 0; o < len[r]; o += kPiece, ++idx)
            if (idx % nparts == part)
                prefetch_l2(M + off[r] + o, (uint32_t)(len[r] - o < kPiece ? len[r] - o : kPiece));
}

// The same loads through L2 only, for a record written earlier in the running
// grid (the read-only path may not see such writes).
template <int FMT>
__device__ __forceinline__ void load_chunk_cg(const uint8_t* M, int R, int C, int rt, int kc, int lane,
                                              Chunk<FMT>& ch) {
    const int KC = C / 64;
    const size_t tile = (size_t)rt * KC + kc;
    if constexpr (FMT == FMT_Q4_0 || FMT == FMT_NVFP4) {
        ch.q = __ldcg(reinterpret_cast<const uint4*>(M + (tile * 32 + lane) * 16));
        ch.sc = __ldcg(reinterpret_cast<const uint2*>(M + (size_t)R * C / 2 + (tile * 8 + (lane >> 2)) * 8));
    } else if constexpr (FMT == FMT_FP8_B128) {
        const size_t qo = (tile * 32 + lane) * 32;
        ch.q0 = __ldcg(reinterpret_cast<const uint4*>(M + qo));
        ch.q1 = __ldcg(reinterpret_cast<const uint4*>(M + qo + 16));
        const int nct = (C + 127) / 128;
        ch.sc = __ldcg(reinterpret_cast<const float*>(M + (size_t)R * C) + (size_t)((rt * 16) / 128) * nct + (kc * 64) / 128);
    } else {
        const size_t qo = (tile * 32 + lane) * 64;
#pragma unroll
        for (int i = 0; i < 4; ++i) ch.q[i] = __ldcg(reinterpret_cast<const uint4*>(M + qo + 16 * i));
    }
}

// The bytes of a matrix that no lane's chunk covers (block-FP8 tile scales and
// the padding up to the 16-byte matrix stride), copied by one CTA per matrix.
template <int FMT>
__device__ __forceinline__ void copy_matrix_tail(const uint8_t* M, uint8_t* D, int R, int C, int tid, int nthr) {
    const size_t begin = FMT == FMT_FP8_B128 ? (size_t)R * C : matrix_bytes(FMT, R, C);
    const size_t end = matrix_stride(FMT, R, C);
    for (size_t i = begin + (size_t)tid * 4; i < end; i += (size_t)nthr * 4)
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
        // A = code * 2^-14 (its bits, e2m1x2_bits_2m14) times scale * 2^7:
        // code * scale * 2^-7, exact in fp16 (at most 6 significant bits, and at
        // least 2^-17 when not zero); the chunk's sum is scaled back by 2^7,
        // exactly, as it is added
        const uint32_t w[4] = {ch.q.x, ch.q.y, ch.q.z, ch.q.w};
        const __half2 k7 = __float2half2_rn(128.0f);
        float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint32_t scw = s < 2 ? ch.sc.x : ch.sc.y;
            const __half2 sh = __hmul2(u32_as_h2(e4m3x2_to_h2((scw >> (16 * (s & 1))) & 0xffffu)), k7);
            const __half2 sg = __low2half2(sh), s8 = __high2half2(sh);
            uint32_t a[4];
            a[0] = h2_as_u32(__hmul2(u32_as_h2(e2m1x2_bits_2m14(w[s])), sg));
            a[1] = h2_as_u32(__hmul2(u32_as_h2(e2m1x2_bits_2m14(w[s] >> 4)), s8));
            a[2] = h2_as_u32(__hmul2(u32_as_h2(e2m1x2_bits_2m14(w[s] >> 8)), sg));
            a[3] = h2_as_u32(__hmul2(u32_as_h2(e2m1x2_bits_2m14(w[s] >> 12)), s8));
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_f16(t, a, b[nb][s][0], b[nb][s][1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = fmaf(128.0f, t[i], acc[i]);
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

// Writes the activation a of (pair, row i) and folds |a| into the pair's
// maximum for the down projection's prescale. The lanes of a warp hold four
// rows of the eight columns lane & 7 (the gate/up epilogue layout); every lane
// of the warp calls it, with pair < 0 where it holds no pair.
template <int FMT>
__device__ __forceinline__ void store_act(const Scratch& s, int pair, int I, int i, float a) {
    if (pair >= 0) s.act[(size_t)pair * I + i] = a;
    if constexpr (FMT != FMT_BF16) {
        unsigned m = pair >= 0 ? __float_as_uint(fabsf(a)) : 0u;
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if ((threadIdx.x & 24) == 0 && pair >= 0) atomicMax(s.act_amax + pair, m);
    }
}

// The prescale of a pair's activations (0 for bf16 experts, whose 16-bit
// parts have fp32's range).
template <int FMT>
__device__ __forceinline__ int pair_act_shift(const Scratch& s, int pair) {
    if constexpr (FMT == FMT_BF16) return 0;
    else return act_shift(__ldcg(s.act_amax + pair));
}

// An fp32 value as two 16-bit parts, hi + lo (fp16, or bf16 for bf16 experts).
template <int FMT>
__device__ __forceinline__ void split_hi_lo(float v, uint16_t& hv, uint16_t& lv) {
    if constexpr (FMT == FMT_BF16) {
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
        hv = *reinterpret_cast<uint16_t*>(&h);
        lv = *reinterpret_cast<uint16_t*>(&l);
    } else {
        __half h = __float2half_rn(v);
        __half l = __float2half_rn(v - __half2float(h));
        hv = *reinterpret_cast<uint16_t*>(&h);
        lv = *reinterpret_cast<uint16_t*>(&l);
    }
}

constexpr int kGUWarps = 8;
constexpr int kDNWarps = 4;
constexpr int kMaxChunksInFlight = 4;

__device__ __forceinline__ void note_miss_start(const Scratch& s, const UnitDesc& d) {
    if (d.dst && threadIdx.x == 0) atomicMin(s.copy_t0, globaltimer_ns());
}
__device__ __forceinline__ void note_miss_end(const Scratch& s, const UnitDesc& d) {
    if (d.dst && threadIdx.x == 0) atomicMax(s.copy_t1, globaltimer_ns());
}

// ---------------------------------------------------------------------------
// Down projection of a decode call by 16-row output tiles over every unit of
// the call. Every pair's activation is staged in shared memory once, split
// into hi + lo 16-bit parts; warps take (unit, group of kDRChunks chunks)
// items with all their weight loads in flight; each item's partial tile goes
// to shared memory per (chunk group, pair, row), and the CTA sums the groups
// in order, weights the picks in rank order and adds the shared expert. No
// partial leaves the SM.
// ---------------------------------------------------------------------------
constexpr int kDRWarps = 16;
constexpr int kDRChunks = 4;

// Shared memory of the row-tile down projection after the U descriptors:
// activations hi and lo [(P + 1)][I + 8] (the last row is zero), partials
// [chunk groups][P][16].
__host__ __device__ inline size_t down_rows_work_bytes(int I, int P) {
    const size_t ld = (size_t)I + 8;
    const int ncg = (I / 64 + kDRChunks - 1) / kDRChunks;
    return 2 * (size_t)(P + 1) * ld * 2 + (size_t)ncg * P * 16 * 4;
}

__host__ __device__ inline size_t down_rows_smem(int I, int KC, int U, int P) {
    (void)KC;
    return (size_t)U * sizeof(UnitDesc) + down_rows_work_bytes(I, P);
}

// Stages the P activations of the call (fp32, written by the gate/up pass)
// as hi + lo 16-bit parts of the prescaled values, plus the zero row, and the
// pairs' prescales in psh [P]; every thread of the CTA takes part, the caller
// synchronises.
template <int FMT>
__device__ __forceinline__ void down_stage_act(const Scratch& s, int P, int I, uint16_t* ah, uint16_t* al, int* psh) {
    const int ld = I + 8, tid = threadIdx.x, nthr = blockDim.x;
    for (int p = tid; p < P; p += nthr) psh[p] = pair_act_shift<FMT>(s, p);
    __syncthreads();
    const int vpr = I / 4;
    const int nv = P * vpr;
    constexpr int B = 4;
    for (int base = tid; base < nv; base += nthr * B) {
        float4 v[B];
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const int j = base + i * nthr;
            if (j < nv) v[i] = __ldcg(reinterpret_cast<const float4*>(s.act) + j);
        }
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const int j = base + i * nthr;
            if (j < nv) {
                const int pr = j / vpr, cv = j - pr * vpr;
                const float sc = pow2f(-psh[pr]);
                const float av[4] = {v[i].x * sc, v[i].y * sc, v[i].z * sc, v[i].w * sc};
                uint16_t hv[4], lv[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) split_hi_lo<FMT>(av[q], hv[q], lv[q]);
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

// The combine of a 16-row output tile for every token: y = sum_j w[t,j] v_j in
// rank order (an fma chain), v_j = the pick's partial sums over the chunk
// groups in ascending order, plus the shared expert's. One warp per (token,
// row): lane j gathers v_j, lane 0 runs the chain in order, so the result is
// the sequential loop's bit for bit. ps: [chunk groups][P][16]; out: the
// tile's first row of token 0, tokens H apart.
__device__ __forceinline__ void combine_rows(const float* ps, const float* wts, int T, int k, int P, int ncg,
                                             int has_shared, float* __restrict__ out, int H) {
    const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int i = threadIdx.x >> 5; i < T * 16; i += nw) {
        const int t = i >> 4, row = i & 15;
        float v = 0.f;
        if (lane < k || (lane == k && has_shared)) {
            const int pair = lane < k ? t * k + lane : T * k + t;
            for (int cg = 0; cg < ncg; ++cg) v += ps[((size_t)cg * P + pair) * 16 + row];
        }
        float y = 0.f;
        for (int j = 0; j < k; ++j) y = fmaf(wts[t * k + j], __shfl_sync(0xffffffffu, v, j), y);
        const float vs = __shfl_sync(0xffffffffu, v, k < 32 ? k : 0);
        if (has_shared) y += vs;
        if (lane == 0) out[(size_t)t * H + row] = y;
    }
}

// Row tile rt of the output for every token: the units' down projections of
// the staged activations (sd: the call's n_units descriptors in shared
// memory; ps: [chunk groups][P][16] partials), combined with the router
// weights wts. Run by kDRWarps warps; starts and ends with the CTA in step.
template <int FMT>
__device__ void down_rows_tile(const CacheDev& c, const Scratch& s, const UnitDesc* sd, int n_units, int T, int rt,
                               const uint16_t* ah, const uint16_t* al, const int* psh, float* ps, const float* wts,
                               float* __restrict__ out) {
    constexpr int IB = FMT == FMT_BF16 ? 1 : 2;  // items a warp keeps in flight
    const int H = c.H, I = c.I, KC = I / 64, k = c.k;
    const int P = T * k + (c.has_shared ? T : 0);
    const int ld = I + 8;
    const int ncg = (KC + kDRChunks - 1) / kDRChunks;
    const int tid = threadIdx.x, nthr = blockDim.x;
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
            // a missed record was written to its slot by the gate/up pass
            if (d.dst) {
#pragma unroll
                for (int i = 0; i < kDRChunks; ++i) {
                    const int kc = cg * kDRChunks + i;
                    if (kc < KC) load_chunk_cg<FMT>(W, H, I, rt, kc, lane, ch[b][i]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < kDRChunks; ++i) {
                    const int kc = cg * kDRChunks + i;
                    if (kc < KC) load_chunk<FMT>(W, nullptr, H, I, rt, kc, lane, ch[b][i]);
                }
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
                    if (n0 > 0) load_chunk_cg<FMT>(reinterpret_cast<const uint8_t*>(d.dst ? d.dst : d.src) +
                                                       2 * matrix_stride(FMT, I, H), H, I, rt, kc, lane, ch[b][i]);
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
                            ps[((size_t)cg * P + pair) * 16 + g + 8 * h2] = acc[2 * h2 + c2] * gd * pow2f(psh[pair]);
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    combine_rows(ps, wts, T, k, P, ncg, c.has_shared, out + (size_t)rt * 16, H);
    __syncthreads();
}

}  // namespace moe
