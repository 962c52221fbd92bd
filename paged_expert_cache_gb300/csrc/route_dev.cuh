// route_dev.cuh -- device routines of routing and planning, shared by the
// routing kernels (route.cu) and the fused decode-layer kernel (layer.cu).
//
// Router and top-k follow "Your GPU holds 24 GB. This model is 94 GB. It
// still runs." (cloudmash.blog), "The model that should not fit": every
// expert gets a logit, a token keeps its top_k; ties go to the lower expert
// id. The plan is the cache transaction of the same page's section "Inside
// llama.cpp PR #29887: slot maps, banks, and only the misses cross PCIe",
// restated with a last-use clock per slot instead of a linked list: touching
// a slot stamps it with the next clock value, the least recently used slot is
// the one with the smallest stamp. The two give the same victims in the same
// order (initial stamps 0..K-1 put slot 0 at the head).
//
// Bit-exact top-k. Logits are accumulated per lane with an error-free
// two-sum, so each logit is a normalized float pair (hi, lo) carrying ~48
// bits, with a rigorous bound on its distance from the fp64, ascending-index
// sum that defines it. Pairs compare exactly (hi first, then lo) and all the
// ranking arithmetic stays in fp32: fp64 is slow on this part. Only when the
// bounds cannot separate the ranking are the candidates recomputed in the
// definition's own order (sequential fp64, no fused multiply-add) and ranked
// again.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;  // experts per CTA, one warp each
constexpr int kRouteTokens = 8;                  // tokens per CTA

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// (a + b) as a normalized pair: s = RN(a + b), e = a + b - s exactly.
__device__ __forceinline__ float2 norm_pair(float a, float b) {
    float s, e;
    two_sum(a, b, s, e);
    return make_float2(s, e);
}

// Copies n elements global -> shared with every thread's loads of a batch
// in flight before its stores, so the copy costs one round trip per batch
// instead of one per element.
template <typename T, int B = 8>
__device__ __forceinline__ void stage(T* dst, const T* src, int n, int tid, int nthr) {
    for (int base = tid; base < n; base += nthr * B) {
        T v[B];
#pragma unroll
        for (int i = 0; i < B; ++i)
            if (base + i * nthr < n) v[i] = __ldcg(src + base + i * nthr);
#pragma unroll
        for (int i = 0; i < B; ++i)
            if (base + i * nthr < n) dst[base + i * nthr] = v[i];
    }
}

// The same for data other CTAs of the running grid wrote (read through L2).
template <typename T, int B = 8>
__device__ __forceinline__ void stage_cg(T* dst, const T* src, int n, int tid, int nthr) {
    for (int base = tid; base < n; base += nthr * B) {
        T v[B];
#pragma unroll
        for (int i = 0; i < B; ++i)
            if (base + i * nthr < n) v[i] = __ldcg(src + base + i * nthr);
#pragma unroll
        for (int i = 0; i < B; ++i)
            if (base + i * nthr < n) dst[base + i * nthr] = v[i];
    }
}

// Order-preserving map of a float to an unsigned integer.
__device__ __forceinline__ unsigned ord32(float f) {
    const unsigned u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exact comparison of normalized pairs.
__device__ __forceinline__ bool pair_gt(float2 a, float2 b) { return a.x > b.x || (a.x == b.x && a.y > b.y); }
__device__ __forceinline__ bool pair_eq(float2 a, float2 b) { return a.x == b.x && a.y == b.y; }

constexpr int kRouterMaxVec = 16;  // H <= 4096: a lane's router vectors, all in flight at once

// Router vectors per lane: lane l reads columns l*8 + i*256 .. +7 for
// i < router_nvec(H) while they lie below H (H is a multiple of 64, so the
// last round is partial when H is not a multiple of 256: lanes past the row's
// end skip it).
__host__ __device__ __forceinline__ int router_nvec(int H) { return (H + 255) / 256; }

// The lane's share of router row e: 16-byte vectors lane*8 + i*256 < H.
__device__ __forceinline__ void router_row_load(const uint16_t* w, int e, int H, int lane, uint4 (&wv)[kRouterMaxVec]) {
    const uint16_t* wr = w + (size_t)e * H;
    const int nvec = router_nvec(H);
#pragma unroll
    for (int i = 0; i < kRouterMaxVec; ++i)
        if (i < nvec && lane * 8 + i * 256 < H) wv[i] = __ldg(reinterpret_cast<const uint4*>(wr + lane * 8 + i * 256));
}

// The longest chain of roundings a lane's logit sum goes through: its eight
// products per vector, then the five butterfly levels and the bias (with
// room to spare); the error bounds below take it as n.
__device__ __forceinline__ float router_chain(int H) { return (float)(8 * router_nvec(H) + 16); }

// Logits of expert e for tokens t0 .. t0+nt-1 (staged bf16 in xs, [NT][H]),
// one warp, with their bounds; row_vec(i, cb) gives the lane's i-th router
// vector (columns cb .. cb + 7). Each lane sums its own columns in order with
// an error-free two-sum, then the lanes combine in a fixed butterfly, so the
// pair does not depend on which CTA or warp computes it.
template <int NT, class RowVec>
static __device__ void router_logits_warp_f(const CacheDev& c, const RouteArgs& a, const uint16_t* xs, int t0, int nt,
                                            int e, RowVec&& row_vec, float2* logits, float* bounds) {
    const int H = c.H, E = c.E, lane = threadIdx.x & 31;
    float hi[NT], lo[NT], ab[NT];
#pragma unroll
    for (int tt = 0; tt < NT; ++tt) hi[tt] = lo[tt] = ab[tt] = 0.f;
    const int nvec = router_nvec(H);
#pragma unroll
    for (int i = 0; i < kRouterMaxVec; ++i) {
        if (i >= nvec) break;
        const int cb = lane * 8 + i * 256;
        if (cb >= H) continue;  // the partial last round
        const uint4 wvi = row_vec(i, cb);
        float wf[8] = {bf16_lo(wvi.x), bf16_hi(wvi.x), bf16_lo(wvi.y), bf16_hi(wvi.y),
                       bf16_lo(wvi.z), bf16_hi(wvi.z), bf16_lo(wvi.w), bf16_hi(wvi.w)};
#pragma unroll
        for (int tt = 0; tt < NT; ++tt) {
            if (NT == 1 || tt < nt) {
                uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)tt * H + cb);
                float xf[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                               bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float p = __fmul_rn(xf[j], wf[j]);  // exact: two 8-bit significands
                    float sum, err;
                    two_sum(hi[tt], p, sum, err);
                    hi[tt] = sum;
                    lo[tt] = __fadd_rn(lo[tt], err);
                    ab[tt] = __fadd_rn(ab[tt], fabsf(p));
                }
            }
        }
    }
    // butterfly over lanes; every lane ends with the same pair
#pragma unroll
    for (int off = 16; off; off >>= 1) {
#pragma unroll
        for (int tt = 0; tt < NT; ++tt) {
            float oh = __shfl_xor_sync(0xffffffffu, hi[tt], off);
            float ol = __shfl_xor_sync(0xffffffffu, lo[tt], off);
            float oa = __shfl_xor_sync(0xffffffffu, ab[tt], off);
            float sum, err;
            two_sum(hi[tt], oh, sum, err);
            hi[tt] = sum;
            lo[tt] = __fadd_rn(__fadd_rn(lo[tt], ol), err);
            ab[tt] = __fadd_rn(ab[tt], oa);
        }
    }
    if (lane < nt) {
        // Bound, all in fp32: the float-pair sum is within g^2 * S of the
        // exact sum (g = n u / (1 - n u), n the longest chain of roundings,
        // u = 2^-24, S = sum |x w|); the fp64 definition is within
        // H * 2^-52 * S of it plus its own bias rounding (2^-52 |z|); folding
        // the bias into the pair costs at most 2^-46 |z|. Doubled, then
        // rounded up.
        const float n = router_chain(H);
        const float g = n * 0x1p-24f / (1.0f - n * 0x1p-24f);
        float hv = hi[0], lv = lo[0], av = ab[0];
#pragma unroll
        for (int tt = 1; tt < NT; ++tt)
            if (lane == tt) { hv = hi[tt]; lv = lo[tt]; av = ab[tt]; }
        float2 z = norm_pair(hv, lv);
        if (a.bias) {
            float sh, se;
            two_sum(z.x, a.bias[e], sh, se);
            z = norm_pair(sh, __fadd_rn(se, z.y));
        }
        const float S = av * (1.0f + 2.0f * g);
        const float beta = (2.0f * (g * g * S + (float)H * 0x1p-52f * S + 0x1p-44f * fabsf(z.x)) +
                            (float)H * 0x1p-126f * 0x1p-22f) * (1.0f + 0x1p-20f);
        logits[(size_t)(t0 + lane) * E + e] = z;
        bounds[(size_t)(t0 + lane) * E + e] = beta;
    }
}

// Logits of expert e for tokens t0 .. t0+nt-1 (staged bf16 in xs, [NT][H]),
// one warp, with their bounds: the lane's router vectors held in registers
// (wv, loaded by router_row_load) ...
template <int NT>
static __device__ void router_logits_warp(const CacheDev& c, const RouteArgs& a, const uint16_t* xs, int t0, int nt, int e,
                                          const uint4 (&wv)[kRouterMaxVec], float2* logits, float* bounds) {
    router_logits_warp_f<NT>(c, a, xs, t0, nt, e, [&](int i, int) { return wv[i]; }, logits, bounds);
}

// ... or read from the router row staged in shared memory (row: its first
// element): the same vectors, sums and bounds.
template <int NT>
static __device__ void router_logits_warp_smem(const CacheDev& c, const RouteArgs& a, const uint16_t* xs, int t0, int nt,
                                               int e, const uint16_t* row, float2* logits, float* bounds) {
    router_logits_warp_f<NT>(
        c, a, xs, t0, nt, e, [&](int, int cb) { return *reinterpret_cast<const uint4*>(row + cb); }, logits, bounds);
}

// The same logit and bound for one token, with the router row staged in
// shared memory (row: the row's first element, this lane reading vectors
// lane*8 + i*256 as router_logits_warp does) and a rolled loop over the
// vectors: the same operations in the same order, so the same pair and bound,
// from a short instruction stream (code that runs once per call is fetched
// once per call).
static __device__ void router_logit_row(const CacheDev& c, const RouteArgs& a, const uint16_t* xs, const uint16_t* row,
                                        int t, int e, float2* logits, float* bounds) {
    const int H = c.H, E = c.E, lane = threadIdx.x & 31;
    float hi = 0.f, lo = 0.f, ab = 0.f;
    const int nvec = router_nvec(H);
#pragma unroll 1
    for (int i = 0; i < nvec; ++i) {
        const int cb = lane * 8 + i * 256;
        if (cb >= H) break;  // the partial last round
        const uint4 wq = *reinterpret_cast<const uint4*>(row + cb);
        const uint4 xv = *reinterpret_cast<const uint4*>(xs + cb);
        const float wf[8] = {bf16_lo(wq.x), bf16_hi(wq.x), bf16_lo(wq.y), bf16_hi(wq.y),
                             bf16_lo(wq.z), bf16_hi(wq.z), bf16_lo(wq.w), bf16_hi(wq.w)};
        const float xf[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                             bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float p = __fmul_rn(xf[j], wf[j]);
            float sum, err;
            two_sum(hi, p, sum, err);
            hi = sum;
            lo = __fadd_rn(lo, err);
            ab = __fadd_rn(ab, fabsf(p));
        }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        float oh = __shfl_xor_sync(0xffffffffu, hi, off);
        float ol = __shfl_xor_sync(0xffffffffu, lo, off);
        float oa = __shfl_xor_sync(0xffffffffu, ab, off);
        float sum, err;
        two_sum(hi, oh, sum, err);
        hi = sum;
        lo = __fadd_rn(__fadd_rn(lo, ol), err);
        ab = __fadd_rn(ab, oa);
    }
    if (lane == 0) {
        // the bound of router_logits_warp
        const float n = router_chain(H);
        const float g = n * 0x1p-24f / (1.0f - n * 0x1p-24f);
        float2 z = norm_pair(hi, lo);
        if (a.bias) {
            float sh, se;
            two_sum(z.x, a.bias[e], sh, se);
            z = norm_pair(sh, __fadd_rn(se, z.y));
        }
        const float S = ab * (1.0f + 2.0f * g);
        const float beta = (2.0f * (g * g * S + (float)H * 0x1p-52f * S + 0x1p-44f * fabsf(z.x)) +
                            (float)H * 0x1p-126f * 0x1p-22f) * (1.0f + 0x1p-20f);
        logits[(size_t)t * E + e] = z;
        bounds[(size_t)t * E + e] = beta;
    }
}

// Largest |bf16| bit pattern of a token row of H values staged in shared
// memory, by one warp (every lane returns it).
__device__ __forceinline__ unsigned token_absmax_warp(const uint16_t* row, int H, int lane) {
    unsigned m = 0u;
    const uint32_t* r32 = reinterpret_cast<const uint32_t*>(row);
    for (int i = lane; i < H / 2; i += 32) m = max(m, bf16x2_absmax(r32[i]));
    return __reduce_max_sync(0xffffffffu, m);
}

// Logits of one CTA's experts for one CTA's NT tokens, with their bounds.
// tok_shift (or null): the CTAs of the first expert column write the
// fp16 prescale of their tokens there (token_shift), for the expert kernels.
template <int NT>
static __device__ void router_logits_tile(const CacheDev& c, const RouteArgs& a, uint8_t* smem, float2* logits,
                                   float* bounds, int* tok_shift) {
    const int H = c.H, E = c.E;
    const int t0 = blockIdx.y * NT;
    const int nt = min(NT, a.T - t0);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);  // [NT][H]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kRouteWarps + warp;
    uint4 wv[kRouterMaxVec];
    if (e < E) router_row_load(a.w, e, H, lane, wv);  // in flight while the tokens are staged
    const int vec_per_row = H / 8;
    for (int i = threadIdx.x; i < nt * vec_per_row; i += blockDim.x) {
        int tt = i / vec_per_row, cv = i - tt * vec_per_row;
        reinterpret_cast<uint4*>(xs + (size_t)tt * H)[cv] =
            reinterpret_cast<const uint4*>(a.x + (size_t)(t0 + tt) * H)[cv];
    }
    __syncthreads();
    if (tok_shift && blockIdx.x == 0)
        for (int tt = warp; tt < nt; tt += kRouteWarps) {
            const unsigned m = token_absmax_warp(xs + (size_t)tt * H, H, lane);
            if (lane == 0) tok_shift[t0 + tt] = token_shift(m);
        }
    if (e >= E) return;
    router_logits_warp<NT>(c, a, xs, t0, nt, e, wv, logits, bounds);
}

// The logit of (t, e) exactly as the definition states it: fp64, ascending
// h, a product then an add at every step, then the bias.
static __device__ double exact_logit(const RouteArgs& a, int H, int t, int e) {
    const uint16_t* xr = a.x + (size_t)t * H;
    const uint16_t* wr = a.w + (size_t)e * H;
    double acc = 0.0;
    for (int h = 0; h < H; ++h) {
        double xv = (double)__uint_as_float((uint32_t)xr[h] << 16);
        double wv = (double)__uint_as_float((uint32_t)wr[h] << 16);
        acc = __dadd_rn(acc, __dmul_rn(xv, wv));
    }
    if (a.bias) acc = __dadd_rn(acc, (double)a.bias[e]);
    return acc;
}

__device__ __forceinline__ bool better(double za, int ea, double zb, int eb) {
    return za > zb || (za == zb && ea < eb);
}

__device__ __forceinline__ bool better_pair(float2 za, int ea, float2 zb, int eb) {
    return pair_gt(za, zb) || (pair_eq(za, zb) && ea < eb);
}

__device__ __forceinline__ float2 shfl_pair(float2 v, int off) {
    return make_float2(__shfl_xor_sync(0xffffffffu, v.x, off), __shfl_xor_sync(0xffffffffu, v.y, off));
}

// Per-warp shared memory of the ranking: E entries of each array plus the
// k picks. The rounds below are rolled loops over these arrays: the kernel
// runs this code once per call, so a short instruction stream matters more
// than register-resident picks.
struct TopkSmem {
    float2* z;    // logit pairs
    float* b;     // bounds
    int* cand;    // re-rank candidates
    double* z64;  // exact logits of the candidates
    int* sel;     // [kMaxTopK] picks in rank order
    float2* selz; // [kMaxTopK] their logit pairs
    float* selb;  // [kMaxTopK] their bounds
};

__host__ __device__ inline size_t topk_bytes_per_warp(int E) {
    return (size_t)E * (sizeof(float2) + sizeof(float) + sizeof(int) + sizeof(double)) +
           (size_t)kMaxTopK * (sizeof(int) + sizeof(float2) + sizeof(float));
}

__device__ inline TopkSmem topk_layout(uint8_t* base, int E) {
    TopkSmem t;
    t.z64 = reinterpret_cast<double*>(base);
    t.z = reinterpret_cast<float2*>(base + (size_t)E * 8);
    t.selz = reinterpret_cast<float2*>(base + (size_t)E * 16);
    t.b = reinterpret_cast<float*>(base + (size_t)E * 16 + kMaxTopK * 8);
    t.cand = reinterpret_cast<int*>(base + (size_t)E * 20 + kMaxTopK * 8);
    t.sel = reinterpret_cast<int*>(base + (size_t)E * 24 + kMaxTopK * 8);
    t.selb = reinterpret_cast<float*>(base + (size_t)E * 24 + kMaxTopK * 12);
    return t;
}

// Weights of a ranking (picks in w.sel / w.selz, rank order), one warp: the
// softmax over the picks (norm_topk) or over all experts. Every ranking path
// ends here, so a token's weights do not depend on the path that ranked it.
static __device__ __forceinline__ void topk_weights(const CacheDev& c, int t, const TopkSmem& w, int* ids_out,
                                                    float* wts_out) {
    const int E = c.E, k = c.k, lane = threadIdx.x & 31;
    float zref = -INFINITY, sum = 0.f;
    if (!c.norm_topk) {
        for (int e = lane; e < E; e += 32) zref = fmaxf(zref, w.z[e].x);
#pragma unroll
        for (int off = 16; off; off >>= 1) zref = fmaxf(zref, __shfl_xor_sync(0xffffffffu, zref, off));
        for (int e = lane; e < E; e += 32) sum += expf(w.z[e].x - zref);
#pragma unroll
        for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    } else {
        // every lane takes the picks' largest logit and sums their
        // exponentials in rank order: k reads, no cross-lane steps
        for (int j = 0; j < k; ++j) zref = fmaxf(zref, w.selz[j].x);
        for (int j = 0; j < k; ++j) sum += expf(w.selz[j].x - zref);
    }
    if (lane < k) {
        ids_out[t * k + lane] = w.sel[lane];
        wts_out[t * k + lane] = expf(w.selz[lane].x - zref) / sum;
    }
    __syncwarp();
}

// Top-k of token t by one warp; writes ids and weights of the token.
// The scratch comes as its base address (topk_layout's), not as a TopkSmem:
// a reference would put the caller's TopkSmem in local memory, and every
// read of its pointers on the fast path would go there.
static __device__ __noinline__ void topk_token(const CacheDev& c, const Scratch& s, const RouteArgs& a, int t,
                                               uint8_t* wbase, int* rerank_flag, int* ids_out, float* wts_out) {
    const int E = c.E, k = c.k, lane = threadIdx.x & 31;
    const TopkSmem w = topk_layout(wbase, E);
    stage_cg<float2>(w.z, s.logits + (size_t)t * E, E, lane, 32);
    stage_cg<float>(w.b, s.bounds + (size_t)t * E, E, lane, 32);
    __syncwarp();
    // k rounds of argmax over the untaken experts; bit m of `taken` is e = lane + 32 m
    unsigned taken = 0;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
        float2 bz = make_float2(-INFINITY, 0.f);
        int be = 0x7fffffff;
        for (int e = lane, m = 0; e < E; e += 32, ++m)
            if (!((taken >> m) & 1u) && better_pair(w.z[e], e, bz, be)) { bz = w.z[e]; be = e; }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            float2 oz = shfl_pair(bz, off);
            int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (better_pair(oz, oe, bz, be)) { bz = oz; be = oe; }
        }
        if (lane == 0) { w.sel[j] = be; w.selz[j] = bz; }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
    }
    // largest upper bound (z + b, as a pair) over the experts not picked
    float2 mx = make_float2(-INFINITY, 0.f);
    for (int e = lane, m = 0; e < E; e += 32, ++m)
        if (!((taken >> m) & 1u)) {
            float2 up = norm_pair(w.z[e].x, __fadd_ru(w.z[e].y, w.b[e]));
            if (pair_gt(up, mx)) mx = up;
        }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        float2 o = shfl_pair(mx, off);
        if (pair_gt(o, mx)) mx = o;
    }
    __syncwarp();
    // certify: each pick's lower bound is above every later upper bound
    bool ok = true;
    float2 run = mx, lam = make_float2(INFINITY, 0.f);
#pragma unroll 1
    for (int j = k - 1; j >= 0; --j) {
        const float2 zj = w.selz[j];
        const float bj = w.b[w.sel[j]];
        const float2 lower = norm_pair(zj.x, __fsub_rd(zj.y, bj));
        const float2 upper = norm_pair(zj.x, __fadd_ru(zj.y, bj));
        if (!pair_gt(lower, run)) ok = false;
        if (pair_gt(upper, run)) run = upper;
        if (pair_gt(lam, lower)) lam = lower;
    }
    if (!ok) {
        // candidates: every expert whose upper bound reaches the lowest lower
        // bound of the picks; outside this set no expert can be in the top-k
        int nc = 0;
        for (int base = 0; base < E; base += 32) {
            int e = base + lane;
            bool in = false;
            if (e < E) {
                float2 up = norm_pair(w.z[e].x, __fadd_ru(w.z[e].y, w.b[e]));
                in = !pair_gt(lam, up);
            }
            unsigned bal = __ballot_sync(0xffffffffu, in);
            if (in) w.cand[nc + __popc(bal & ((1u << lane) - 1u))] = e;
            nc += __popc(bal);
        }
        __syncwarp();
        for (int i = lane; i < nc; i += 32) w.z64[i] = exact_logit(a, c.H, t, w.cand[i]);
        __syncwarp();
        // k rounds over the candidates; a picked candidate is marked by
        // storing -1 - e in its cand entry
#pragma unroll 1
        for (int j = 0; j < k; ++j) {
            double bz = -INFINITY;
            int be = 0x7fffffff, bi = -1;
            for (int i = lane; i < nc; i += 32) {
                int e = w.cand[i];
                if (e >= 0 && better(w.z64[i], e, bz, be)) { bz = w.z64[i]; be = e; bi = i; }
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                double oz = __shfl_xor_sync(0xffffffffu, bz, off);
                int oe = __shfl_xor_sync(0xffffffffu, be, off);
                int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (better(oz, oe, bz, be)) { bz = oz; be = oe; bi = oi; }
            }
            if (lane == 0) { w.sel[j] = be; w.selz[j] = w.z[be]; }
            if (lane == (bi & 31)) w.cand[bi] = -1 - be;
            __syncwarp();
        }
        if (lane == 0) *rerank_flag = 1;
    }
    __syncwarp();
    topk_weights(c, t, w, ids_out, wts_out);
}

// Descending bitonic sorting network over NPL (a power of two) keys held in
// registers: every index is a compile-time constant after unrolling.
template <int NPL>
__device__ __forceinline__ void sort_desc(unsigned long long (&key)[NPL]) {
#pragma unroll
    for (int size = 2; size <= NPL; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                const int l = i ^ stride;
                if (l > i) {
                    const unsigned long long a = key[i], b = key[l];
                    const bool swap = ((i & size) == 0) ? (a < b) : (a > b);
                    key[i] = swap ? b : a;
                    key[l] = swap ? a : b;
                }
            }
        }
    }
}

// Certifies the k picks in w.sel / w.selz / w.selb (rank order) against
// their bounds, given mx, the largest upper bound (z + b, as a pair) over the
// experts not picked, and writes the token's ids and weights; where the bounds
// leave the order open, ranks the token again exactly (topk_token). One warp.
static __device__ void topk_certify_finish(const CacheDev& c, const Scratch& s, const RouteArgs& a, int t,
                                           const TopkSmem& w, float2 mx, int* rerank_flag, int* ids_out,
                                           float* wts_out) {
    const int E = c.E, k = c.k, lane = threadIdx.x & 31;
    // certify: lane j checks that pick j's lower bound is above the upper
    // bounds of every later pick and of every expert not picked
    float2 lower = make_float2(-INFINITY, 0.f), sfx = make_float2(-INFINITY, 0.f);
    if (lane < k) {
        const float2 zj = w.selz[lane];
        const float bj = w.selb[lane];
        lower = norm_pair(zj.x, __fsub_rd(zj.y, bj));
        sfx = norm_pair(zj.x, __fadd_ru(zj.y, bj));
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {  // inclusive suffix max over lanes lane..31
        const float2 o = make_float2(__shfl_down_sync(0xffffffffu, sfx.x, off), __shfl_down_sync(0xffffffffu, sfx.y, off));
        if (lane + off < 32 && pair_gt(o, sfx)) sfx = o;
    }
    float2 later = make_float2(__shfl_down_sync(0xffffffffu, sfx.x, 1), __shfl_down_sync(0xffffffffu, sfx.y, 1));
    if (lane == 31 || lane + 1 >= k) later = make_float2(-INFINITY, 0.f);
    if (pair_gt(mx, later)) later = mx;
    const bool ok = __all_sync(0xffffffffu, lane >= k || pair_gt(lower, later));
    if (!ok) {
        topk_token(c, s, a, t, reinterpret_cast<uint8_t*>(w.z64), rerank_flag, ids_out, wts_out);
        return;
    }
    topk_weights(c, t, w, ids_out, wts_out);
}

// Top-k of token t by one warp, from sorted per-lane lists. Lane l holds the
// experts l, l + 32, ... as 64-bit keys: ord(hi) in the high word, then ord(lo)
// with its low ten bits replaced by 1023 - e, so keys are distinct and order
// by hi, then (almost) lo, then the lower expert. Each lane sorts its keys;
// a round is one butterfly max over the lanes' heads, and the lane that owns
// the winner pops it. The picks are then certified against the exact pairs
// and their bounds, in parallel over the picks: where a truncated lo (or the
// bounds) leaves the order open, the token is ranked again by topk_token,
// which re-ranks exactly -- so the result never depends on the truncation.
// Logit pairs and bounds are staged in the warp's TopkSmem for that path.
template <int NPL>
static __device__ __forceinline__ void topk_token_fast(const CacheDev& c, const Scratch& s, const RouteArgs& a, int t,
                                                       const TopkSmem& w, int* rerank_flag, int* ids_out,
                                                       float* wts_out) {
    const int E = c.E, k = c.k, lane = threadIdx.x & 31;
    float2* wz = w.z;
    float* wb = w.b;
    unsigned long long key[NPL];
#pragma unroll
    for (int m = 0; m < NPL; ++m) {
        const int e = lane + 32 * m;
        key[m] = 0ull;
        if (e < E) {
            const float2 z = __ldcg(s.logits + (size_t)t * E + e);
            const float bd = __ldcg(s.bounds + (size_t)t * E + e);
            wz[e] = z;
            wb[e] = bd;
            key[m] = ((unsigned long long)ord32(z.x) << 32) |
                     (unsigned long long)((ord32(__fadd_rn(z.y, 0.0f)) & ~1023u) | (unsigned)(1023 - e));
        }
    }
    sort_desc<NPL>(key);
    __syncwarp();
    for (int j = 0; j < k; ++j) {
        // the largest head over the lanes: its high word by one reduction,
        // then (when heads tie there) its low word among the tied lanes; the
        // keys are distinct, so one lane holds the winner
        const unsigned hi = (unsigned)(key[0] >> 32);
        const unsigned mhi = __reduce_max_sync(0xffffffffu, hi);
        const unsigned tied = __ballot_sync(0xffffffffu, hi == mhi);
        unsigned long long best;
        if (__popc(tied) == 1) {
            best = __shfl_sync(0xffffffffu, key[0], __ffs(tied) - 1);
        } else {
            const unsigned lo = hi == mhi ? (unsigned)key[0] : 0u;
            best = ((unsigned long long)mhi << 32) | __reduce_max_sync(0xffffffffu, lo);
        }
        if (key[0] == best) {
            const int e = 1023 - (int)(best & 1023ull);
            w.sel[j] = e;
            w.selz[j] = wz[e];
            w.selb[j] = wb[e];
#pragma unroll
            for (int m = 0; m + 1 < NPL; ++m) key[m] = key[m + 1];
            key[NPL - 1] = 0ull;
        }
    }
    __syncwarp();
    // largest upper bound (z + b, as a pair) over the experts not picked
    float2 mx = make_float2(-INFINITY, 0.f);
#pragma unroll
    for (int m = 0; m < NPL; ++m) {
        if (key[m]) {
            const int e = 1023 - (int)(key[m] & 1023ull);
            const float2 up = norm_pair(wz[e].x, __fadd_ru(wz[e].y, wb[e]));
            if (pair_gt(up, mx)) mx = up;
        }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        const float2 o = shfl_pair(mx, off);
        if (pair_gt(o, mx)) mx = o;
    }
    topk_certify_finish(c, s, a, t, w, mx, rerank_flag, ids_out, wts_out);
}


// The largest of the lanes' 64-bit keys (all distinct, or zero): the high
// words by one reduction, then, where several lanes tie there, the low words
// among the tied lanes. Every lane of the warp calls it and gets the key.
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long key) {
    const unsigned hi = (unsigned)(key >> 32);
    const unsigned mhi = __reduce_max_sync(0xffffffffu, hi);
    const unsigned tied = __ballot_sync(0xffffffffu, hi == mhi);
    if (__popc(tied) == 1) return __shfl_sync(0xffffffffu, key, __ffs(tied) - 1);
    const unsigned lo = hi == mhi ? (unsigned)key : 0u;
    return ((unsigned long long)mhi << 32) | __reduce_max_sync(0xffffffffu, lo);
}

// Candidates the threshold selection of topk_block_select ranks itself; with
// more it falls back to the sorted-list merge.
constexpr int kBlockCandMax = 128;

// Top-k of token 0 by the whole CTA (E <= blockDim.x <= 32 kMaxTopK, k <=
// kMaxTopK): thread e builds expert e's key (the orderable 64-bit key of
// topk_token_fast: the logit's high part, then its low part with 1023 - e in
// the low bits, so keys are distinct and nonzero).
//   Threshold selection: L, the k-th largest of the warps' largest keys, is
//   at most the k-th largest key overall (k warp maxima are >= L), so every
//   pick has a key >= L. The keys >= L are gathered as candidates (about 16 of
//   512 for random logits); each candidate's rank is the number of candidates
//   above it, which for a pick is its rank among all keys. Ranks below k are
//   the picks, in descending order.
//   With more than kBlockCandMax candidates, the sorted-list merge: each warp
//   takes its k largest keys by k rounds of a warp-wide maximum into wl
//   [warps][kMaxTopK], and warp 0 merges the lists by k rounds over their heads.
// Both give the k largest keys in order. The certificate is topk_token_fast's
// (each pick's lower bound above the upper bound of everything ranked after
// it), checked by every expert against the picks ranked above it and combined
// with one block-wide AND; warp 0 then weighs as topk_token_fast does, or
// re-ranks exactly. Every thread of the CTA calls it; lowb: k entries of shared
// memory; the candidates use w.z64 (E >= kBlockCandMax entries, free until
// the exact re-rank).
static __device__ void topk_block_select(const CacheDev& c, const Scratch& s, const RouteArgs& a, const TopkSmem& w,
                                         unsigned long long* wl, float2* lowb, int* rerank_flag, int* ids_out,
                                         float* wts_out) {
    const int E = c.E, k = c.k, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nw = (int)(blockDim.x >> 5);
    __shared__ unsigned long long wmax[kMaxTopK * 2];
    __shared__ int ncand;
    unsigned long long key = 0ull;
    if (tid < E) {
        const float2 z = __ldcg(s.logits + tid);
        w.z[tid] = z;
        w.b[tid] = __ldcg(s.bounds + tid);
        key = ((unsigned long long)ord32(z.x) << 32) |
              (unsigned long long)((ord32(__fadd_rn(z.y, 0.0f)) & ~1023u) | (unsigned)(1023 - tid));
    }
    {
        const unsigned long long m = warp_max_key(key);
        if (lane == 0) wmax[warp] = m;
        if (tid == 0) ncand = 0;
    }
    __syncthreads();
    // L: the k-th largest warp maximum (lanes past the warps hold zero)
    unsigned long long thr;
    {
        unsigned long long m = lane < nw ? wmax[lane] : 0ull;
        int r = 0;
#pragma unroll 4
        for (int x = 0; x < nw; ++x) r += wmax[x] > m ? 1 : 0;
        // the lane whose maximum has exactly k - 1 larger ones holds L (maxima
        // are distinct but for zeros; with fewer than k nonzero maxima L is 0)
        const unsigned hit = __ballot_sync(0xffffffffu, lane < nw && r == k - 1);
        thr = hit ? __shfl_sync(0xffffffffu, m, __ffs(hit) - 1) : 0ull;
    }
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(w.z64);
    {
        const bool in = key != 0ull && key >= thr;
        const unsigned bal = __ballot_sync(0xffffffffu, in);
        int base = 0;
        if (lane == 0 && bal) base = atomicAdd(&ncand, __popc(bal));
        base = __shfl_sync(0xffffffffu, base, 0);
        const int pos = base + __popc(bal & ((1u << lane) - 1u));
        if (in && pos < kBlockCandMax) cand[pos] = key;
    }
    __syncthreads();
    const int nc = ncand;
    if (nc <= kBlockCandMax) {
        if (tid < nc) {
            const unsigned long long x = cand[tid];
            int rank = 0;
#pragma unroll 4
            for (int u = 0; u < nc; ++u) rank += cand[u] > x ? 1 : 0;
            if (rank < k) {
                const int e = 1023 - (int)(x & 1023ull);
                const float2 ze = w.z[e];
                const float be = w.b[e];
                w.sel[rank] = e;
                w.selz[rank] = ze;
                w.selb[rank] = be;
                lowb[rank] = norm_pair(ze.x, __fsub_rd(ze.y, be));
            }
        }
    } else {
        // 1. each warp's k largest keys, in order (a popped key becomes zero)
        {
            unsigned long long mine = key;
#pragma unroll 1
            for (int j = 0; j < k; ++j) {
                const unsigned long long best = warp_max_key(mine);
                if (lane == 0) wl[warp * kMaxTopK + j] = best;
                if (mine == best) mine = 0ull;
            }
        }
        __syncthreads();
        // 2. warp 0 merges the sorted lists: lane l walks list l
        if (warp == 0) {
            int pos = 0;
            unsigned long long head = lane < nw ? wl[lane * kMaxTopK] : 0ull;
#pragma unroll 1
            for (int j = 0; j < k; ++j) {
                const unsigned long long best = warp_max_key(head);
                if (head == best) {
                    ++pos;
                    head = pos < k ? wl[lane * kMaxTopK + pos] : 0ull;
                }
                if (lane == 0) {
                    const int e = 1023 - (int)(best & 1023ull);
                    const float2 ze = w.z[e];
                    const float be = w.b[e];
                    w.sel[j] = e;
                    w.selz[j] = ze;
                    w.selb[j] = be;
                    lowb[j] = norm_pair(ze.x, __fsub_rd(ze.y, be));
                }
            }
        }
    }
    __syncthreads();
    // 3. Certified when every pick's lower bound lies above the upper bound of
    // every expert ranked after it: each expert checks itself against the
    // picks ranked before it (all k for an expert not picked), and the CTA
    // takes the AND.
    int good = 1;
    if (tid < E) {
        const float2 z = w.z[tid];
        const float2 up = norm_pair(z.x, __fadd_ru(z.y, w.b[tid]));
#pragma unroll 1
        for (int j = 0; j < k && w.sel[j] != tid; ++j) good &= pair_gt(lowb[j], up) ? 1 : 0;
    }
    const int ok = __syncthreads_and(good);
    if (warp == 0) {
        if (ok) topk_weights(c, 0, w, ids_out, wts_out);
        else topk_token(c, s, a, 0, reinterpret_cast<uint8_t*>(w.z64), rerank_flag, ids_out, wts_out);
    }
}

// Top-k of token 0 by the first E threads of the CTA (E <= blockDim.x): thread
// e builds expert e's key (the orderable 64-bit key of topk_token_fast: the
// logit's high part, then its low part with 1023 - e in the low bits, so keys
// are distinct), and its rank is the number of keys above it. Ranks below k
// are the picks, in the same order as the sorted-list rounds give. The
// certificate is topk_token_fast's (each pick's lower bound above the upper
// bound of everything ranked after it), checked by every expert against the
// picks above it and combined with one block-wide AND; warp 0 then weighs as
// topk_token_fast does. Every thread of the CTA calls it; keys: E entries and
// lowb: k entries of shared memory.
static __device__ void topk_rank_block(const CacheDev& c, const Scratch& s, const RouteArgs& a, const TopkSmem& w,
                                       unsigned long long* keys, float2* lowb, int* rerank_flag, int* ids_out,
                                       float* wts_out) {
    const int E = c.E, k = c.k, tid = threadIdx.x, warp = tid >> 5;
    float2 z = make_float2(-INFINITY, 0.f);
    float bd = 0.f;
    unsigned long long key = 0ull;
    if (tid < E) {
        z = __ldcg(s.logits + tid);
        bd = __ldcg(s.bounds + tid);
        w.z[tid] = z;
        w.b[tid] = bd;
        key = ((unsigned long long)ord32(z.x) << 32) |
              (unsigned long long)((ord32(__fadd_rn(z.y, 0.0f)) & ~1023u) | (unsigned)(1023 - tid));
        keys[tid] = key;
    }
    __syncthreads();
    // every expert's upper bound; a pick's lower bound goes to lowb[rank]
    float2 up = make_float2(-INFINITY, 0.f);
    int rank = E;
    if (tid < E) {
        rank = 0;
        const ulonglong2* k2 = reinterpret_cast<const ulonglong2*>(keys);
#pragma unroll 4
        for (int i = 0; i < E / 2; ++i) {
            const ulonglong2 v = k2[i];
            rank += (v.x > key) + (v.y > key);
        }
        if (E & 1) rank += keys[E - 1] > key;
        if (rank < k) {
            w.sel[rank] = tid;
            w.selz[rank] = z;
            w.selb[rank] = bd;
            lowb[rank] = norm_pair(z.x, __fsub_rd(z.y, bd));
        }
        up = norm_pair(z.x, __fadd_ru(z.y, bd));
    }
    __syncthreads();
    // Certified when every pick's lower bound lies above the upper bound of
    // every expert ranked after it: each expert checks itself against the
    // picks ranked before it, and the CTA takes the AND.
    int good = 1;
    if (tid < E) {
        const int nj = rank < k ? rank : k;
        for (int j = 0; j < nj; ++j) good &= pair_gt(lowb[j], up) ? 1 : 0;
    }
    const int ok = __syncthreads_and(good);
    if (warp == 0) {
        if (ok) topk_weights(c, 0, w, ids_out, wts_out);
        else topk_token(c, s, a, 0, reinterpret_cast<uint8_t*>(w.z64), rerank_flag, ids_out, wts_out);
    }
}

__device__ __forceinline__ void topk_dispatch(const CacheDev& c, const Scratch& s, const RouteArgs& a, int t,
                                              const TopkSmem& w, int* rerank_flag, int* ids_out, float* wts_out) {
    if (c.E <= 32) topk_token_fast<1>(c, s, a, t, w, rerank_flag, ids_out, wts_out);
    else if (c.E <= 128) topk_token_fast<4>(c, s, a, t, w, rerank_flag, ids_out, wts_out);
    else if (c.E <= 256) topk_token_fast<8>(c, s, a, t, w, rerank_flag, ids_out, wts_out);
    else if (c.E <= 512) topk_token_fast<16>(c, s, a, t, w, rerank_flag, ids_out, wts_out);
    else topk_token(c, s, a, t, reinterpret_cast<uint8_t*>(w.z64), rerank_flag, ids_out, wts_out);
}

// ---------------------------------------------------------------------------
// Plan of a decode call (T <= 32): the cache transaction, run by one CTA on
// a copy of the pool's state held in shared memory.
// ---------------------------------------------------------------------------
constexpr int kVictimLists = 16;  // misses per call the fast victim search takes (more: one round per miss)

struct PlanSmem {
    unsigned long long* lu;  // [K] last-use stamps of the pool
    int* kof;                // [K] keys of the pool's slots
    int* smap;               // [E] slot map of the layer
    int* first;              // [E] first pair index routed to e
    int* unit_of;            // [E]
    unsigned* missbits;      // [E/32 + 1]
    int* u_expert;           // [U]
    int* u_slot;             // [U]
    int* u_hit;              // [U]
    int* u_cnt;              // [U+1]
    int* p_unit;             // [P]
    int* victims;            // [U]
    int* misses;             // [U] miss experts ascending
    int* ids;                // [T*k] this call's picks
    unsigned long long* wmin;  // [32]
    int* wslot;              // [32]
    unsigned long long* vkey;  // [32][kVictimLists]: each warp's smallest victim keys, in order
    int* vslot;              // [32][kVictimLists]: their slots
    int* scal;               // [8]
    float* gl;               // [(E+1)*3] NVFP4 global scales of the layer (+ shared)
    size_t bytes;
};

__host__ __device__ inline PlanSmem plan_layout(uint8_t* base, int E, int K, int n_ids, int U, int P) {
    PlanSmem m;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* q = base + off;
        off += (bytes + 15) & ~(size_t)15;
        return q;
    };
    m.lu = (unsigned long long*)take(sizeof(unsigned long long) * K);
    m.kof = (int*)take(sizeof(int) * K);
    m.smap = (int*)take(sizeof(int) * E);
    m.first = (int*)take(sizeof(int) * E);
    m.unit_of = (int*)take(sizeof(int) * E);
    m.missbits = (unsigned*)take(sizeof(unsigned) * (E / 32 + 1));
    m.u_expert = (int*)take(sizeof(int) * U);
    m.u_slot = (int*)take(sizeof(int) * U);
    m.u_hit = (int*)take(sizeof(int) * U);
    m.u_cnt = (int*)take(sizeof(int) * (U + 1));
    m.p_unit = (int*)take(sizeof(int) * P);
    m.victims = (int*)take(sizeof(int) * U);
    m.misses = (int*)take(sizeof(int) * U);
    m.ids = (int*)take(sizeof(int) * n_ids);
    m.wmin = (unsigned long long*)take(sizeof(unsigned long long) * 32);
    m.wslot = (int*)take(sizeof(int) * 32);
    m.vkey = (unsigned long long*)take(sizeof(unsigned long long) * 32 * kVictimLists);
    m.vslot = (int*)take(sizeof(int) * 32 * kVictimLists);
    m.scal = (int*)take(sizeof(int) * 8);
    m.gl = (float*)take(sizeof(float) * (E + 1) * 3);
    m.bytes = off;
    return m;
}

static __device__ __noinline__ void write_trace(const CacheDev& c, const Scratch& s, int layer, int T, int n_ids, int n_hit,
                            int n_fill, int n_uniq) {
    // thread 0 only
    unsigned long long idx = *c.trace_count;
    int* r = c.trace + (size_t)(idx % (unsigned long long)c.trace_cap) * c.trace_stride;
    int maxids = (c.trace_stride - 6) / 5;
    int ni = min(n_ids, maxids), nf = min(n_fill, maxids);
    r[0] = layer; r[1] = T; r[2] = ni; r[3] = n_hit; r[4] = nf; r[5] = n_uniq;
    int* p = r + 6;
    for (int i = 0; i < ni; ++i) p[i] = s.ids[i];
    p += ni;
    for (int i = 0; i < ni; ++i) p[i] = s.slot_of[i];
    p += ni;
    for (int i = 0; i < ni; ++i) p[i] = s.hit_of[i];
    p += ni;
    for (int i = 0; i < nf; ++i) p[i] = s.copy_expert[i];
    p += nf;
    for (int i = 0; i < nf; ++i) p[i] = s.copy_slot[i];
    *c.trace_count = idx + 1;
}

// Copies the pool's state into shared memory; run by threads tid of nthr
// (the warps that are not ranking tokens, when there are any).
static __device__ void plan_prefetch(const CacheDev& c, const RouteArgs& a, const PlanSmem& m, int pool, int tid, int nthr,
                              unsigned long long* clk) {
    const unsigned long long* lu = c.last_use + (size_t)pool * c.K;
    const int* kof = c.key_of + (size_t)pool * c.K;
    const int* smap = c.slot_map + (size_t)a.layer * c.E;
    if (tid == 0) *clk = c.clock[pool];
    stage<unsigned long long>(m.lu, lu, c.K, tid, nthr);
    stage<int>(m.kof, kof, c.K, tid, nthr);
    stage<int>(m.smap, smap, c.E, tid, nthr);
    for (int e = tid; e < c.E; e += nthr) m.first[e] = 0x7fffffff;
    if (c.fmt == FMT_NVFP4) {
        stage<float>(m.gl, c.gtable + (size_t)a.layer * c.E * 3, c.E * 3, tid, nthr);
        if (tid < 3) m.gl[c.E * 3 + tid] = c.gtable[((size_t)c.L * c.E + a.layer) * 3 + tid];
    }
    for (int i = tid; i <= c.E / 32; i += nthr) m.missbits[i] = 0u;
}

// LFU victim order (eviction MOE_EVICT_LFU): the staged last-use stamps are
// replaced in shared memory by 64-bit keys, (uses of the slot's key + 1, or 0
// for an empty slot) above the stamp's low 40 bits, so the smallest keys are
// empty slots first, then the fewest uses, then the least recent. The slots
// this call holds (stamped from clk on) become ~0 and are never chosen.
constexpr unsigned kLfuUseCap = 1u << 23;
__device__ __forceinline__ void lfu_victim_keys(const CacheDev& c, const PlanSmem& m, unsigned long long clk) {
    for (int i = threadIdx.x; i < c.K; i += blockDim.x) {
        const unsigned long long st = m.lu[i];
        if (st >= clk) {
            m.lu[i] = ~0ull;
            continue;
        }
        const int key = m.kof[i];
        unsigned long long u = 0ull;
        if (key >= 0) {
            const unsigned n = c.uses[key];
            u = (unsigned long long)(n < kLfuUseCap ? n : kLfuUseCap) + 1ull;
        }
        m.lu[i] = (u << 40) | (st & ((1ull << 40) - 1ull));
    }
    __syncthreads();
}

// The smallest of the lanes' 64-bit keys (the same pattern as warp_max_key).
__device__ __forceinline__ unsigned long long warp_min_key(unsigned long long key) {
    const unsigned hi = (unsigned)(key >> 32);
    const unsigned mhi = __reduce_min_sync(0xffffffffu, hi);
    const unsigned tied = __ballot_sync(0xffffffffu, hi == mhi);
    if (__popc(tied) == 1) return __shfl_sync(0xffffffffu, key, __ffs(tied) - 1);
    const unsigned lo = hi == mhi ? (unsigned)key : 0xffffffffu;
    return ((unsigned long long)mhi << 32) | __reduce_min_sync(0xffffffffu, lo);
}

// The nmiss (<= kVictimLists) slots of the pool with the smallest keys, in
// ascending order, into m.victims: the least recently used slots (keys are
// the last-use stamps) or the LFU order (lfu_victim_keys). Keys are distinct,
// except the ~0 of slots the call holds, which never rank among the nmiss
// smallest. A threshold selection (below) takes the usual case; otherwise
// thread t scans slots t, t + nthr, ... (at most 64 of them); each
// warp takes its nmiss smallest keys by nmiss rounds of a warp-wide minimum,
// where the winning lane then looks for its next smallest, into m.vkey /
// m.vslot; warp 0 merges the warps' sorted lists the same way. The same
// victims, in the same order, as nmiss rounds of a block-wide minimum. Every
// thread of the block calls it.
__device__ __forceinline__ void select_victims(const PlanSmem& m, int K, int nmiss) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
    // Threshold selection first: U, the nmiss-th smallest of the warps'
    // smallest keys, is at least the nmiss-th smallest key (nmiss warp minima
    // are <= U), so the victims are among the keys <= U (a few for LRU
    // stamps); each such candidate's rank is the number of candidates below it
    // (keys are distinct). Small pools (under two keys per thread: the rounds
    // are cheap there), too many candidates (ties at ~0) or more misses than
    // warps: the rounds below.
    if (K >= 2 * nthr) {
        constexpr int kCandMax = 128;
        __shared__ unsigned long long wmin[32];
        __shared__ int ncand;
        unsigned long long mn = ~0ull;
        for (int i = tid; i < K; i += nthr) mn = min(mn, m.lu[i]);
        const unsigned long long wm = warp_min_key(mn);
        if (lane == 0) wmin[warp] = wm;
        if (tid == 0) ncand = 0;
        __syncthreads();
        int nc = kCandMax + 1;
        if (nmiss <= nw) {
            const unsigned long long mine = lane < nw ? wmin[lane] : ~0ull;
            int r = 0;
            for (int x = 0; x < nw; ++x) r += wmin[x] < mine ? 1 : 0;
            const unsigned hit = __ballot_sync(0xffffffffu, lane < nw && r == nmiss - 1);
            const unsigned long long u = hit ? __shfl_sync(0xffffffffu, mine, __ffs(hit) - 1) : ~0ull;
            for (int i0 = 0; i0 < K; i0 += nthr) {
                const int i = i0 + tid;
                const bool in = i < K && m.lu[i] <= u;
                const unsigned bal = __ballot_sync(0xffffffffu, in);
                int base = 0;
                if (lane == 0 && bal) base = atomicAdd(&ncand, __popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                const int pos = base + __popc(bal & ((1u << lane) - 1u));
                if (in && pos < kCandMax) {
                    m.vkey[pos] = m.lu[i];
                    m.vslot[pos] = i;
                }
            }
            __syncthreads();
            nc = ncand;
        }
        if (nc <= kCandMax) {
            if (tid < nc) {
                const unsigned long long x = m.vkey[tid];
                int rank = 0;
                for (int y = 0; y < nc; ++y) rank += m.vkey[y] < x ? 1 : 0;
                if (rank < nmiss) m.victims[rank] = m.vslot[tid];
            }
            __syncthreads();
            return;
        }
        __syncthreads();  // the rounds below rewrite vkey / vslot
    }
    unsigned long long taken = 0ull;  // bit r: slot tid + r * nthr is already a victim
    unsigned long long v = ~0ull;
    int sl = -1;
    auto next_smallest = [&]() {
        v = ~0ull;
        sl = -1;
        int r = 0;
        for (int i = tid; i < K; i += nthr, ++r)
            if (!((taken >> r) & 1ull) && m.lu[i] < v) {
                v = m.lu[i];
                sl = i;
            }
    };
    next_smallest();
#pragma unroll 1
    for (int j = 0; j < nmiss; ++j) {
        const unsigned long long best = warp_min_key(v);
        const unsigned win = __ballot_sync(0xffffffffu, v == best && sl >= 0);
        const int wlane = win ? __ffs(win) - 1 : 0;
        const int bsl = __shfl_sync(0xffffffffu, sl, wlane);
        if (lane == 0) {
            m.vkey[warp * kVictimLists + j] = win ? best : ~0ull;
            m.vslot[warp * kVictimLists + j] = win ? bsl : -1;
        }
        if (win && lane == wlane) {
            taken |= 1ull << ((bsl - tid) / nthr);
            next_smallest();
        }
    }
    __syncthreads();
    if (warp == 0) {
        int pos = 0;
        unsigned long long head = lane < nw ? m.vkey[lane * kVictimLists] : ~0ull;
#pragma unroll 1
        for (int j = 0; j < nmiss; ++j) {
            const unsigned long long best = warp_min_key(head);
            const unsigned win = __ballot_sync(0xffffffffu, head == best && lane < nw);
            const int wlane = __ffs(win) - 1;
            if (lane == wlane) {
                m.victims[j] = m.vslot[lane * kVictimLists + pos];
                ++pos;
                head = pos < nmiss ? m.vkey[lane * kVictimLists + pos] : ~0ull;
            }
        }
    }
    __syncthreads();
}

// ids_in: the call's picks ([T][k]). The descriptors go to units_out
// (global for the expert kernels, or the CTA's shared memory when every CTA
// plans for itself). Only a committing CTA writes the pool's state, the fill
// list, the per-pick slots, the stats and the trace.
static __device__ void plan_decode(const CacheDev& c, const Scratch& s, const RouteArgs& a, const PlanSmem& m,
                            unsigned long long clk, const int* ids_in, UnitDesc* units_out, bool commit) {
    const int E = c.E, k = c.k, T = a.T, layer = a.layer;
    const int n_ids = T * k;
    const int pool = c.pool_mode ? 0 : layer;
    const int K = c.K;
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int P = n_ids + (c.has_shared ? T : 0);
    int* g_slot_map = c.slot_map + (size_t)layer * E;
    int* g_key_of = c.key_of + (size_t)pool * K;
    unsigned long long* g_last_use = c.last_use + (size_t)pool * K;

    // 1. dedupe: first occurrence in [token][rank] order
    for (int i = tid; i < n_ids; i += nthr) {
        int e = ids_in[i];
        m.ids[i] = e;
        atomicMin(&m.first[e], i);
    }
    __syncthreads();
    if (tid < 32) {
        int base = 0;
        for (int i0 = 0; i0 < n_ids; i0 += 32) {
            int i = i0 + tid;
            bool f = i < n_ids && m.first[m.ids[i]] == i;
            unsigned bal = __ballot_sync(0xffffffffu, f);
            if (f) {
                int u = base + __popc(bal & ((1u << tid) - 1u));
                m.unit_of[m.ids[i]] = u;
                m.u_expert[u] = m.ids[i];
            }
            base += __popc(bal);
        }
        __syncwarp();
        const int nu = base;
        // every expert of the call counts one more use (LFU)
        if (commit && c.lfu)
            for (int u = tid; u < nu; u += 32) c.uses[(size_t)layer * E + m.u_expert[u]] += 1u;
        // 2. hits, touched in unit order: stamps clock + hit rank
        int hb = 0;
        for (int u0 = 0; u0 < nu; u0 += 32) {
            int u = u0 + tid;
            int sl = u < nu ? m.smap[m.u_expert[u]] : -1;
            bool h = sl >= 0;
            unsigned bal = __ballot_sync(0xffffffffu, h);
            if (u < nu) {
                m.u_hit[u] = h;
                m.u_slot[u] = sl;
                if (h) {
                    unsigned long long st = clk + hb + __popc(bal & ((1u << tid) - 1u));
                    m.lu[sl] = st;
                    if (commit) g_last_use[sl] = st;
                } else {
                    atomicOr(&m.missbits[m.u_expert[u] >> 5], 1u << (m.u_expert[u] & 31));
                }
            }
            hb += __popc(bal);
        }
        __syncwarp();
        // misses in ascending expert order
        int mb = 0;
        for (int w0 = 0; w0 <= E / 32; w0 += 32) {
            int wi = w0 + tid;
            unsigned bits = wi <= E / 32 ? m.missbits[wi] : 0u;
            int cnt = __popc(bits);
            int incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (tid >= off) incl += v;
            }
            int pos = mb + incl - cnt;
            while (bits) {
                int b = __ffs(bits) - 1;
                bits &= bits - 1;
                m.misses[pos++] = wi * 32 + b;
            }
            mb += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (tid == 0) {
            m.scal[0] = nu;
            m.scal[1] = hb;
        }
    }
    __syncthreads();
    const int nu = m.scal[0];
    const int nh = m.scal[1];
    const int nmiss = nu - nh;
    if (c.lfu && nmiss > 0) lfu_victim_keys(c, m, clk);
    // 3. victims: the nmiss smallest stamps of the pool (LFU: keys), smallest first
    if (nmiss > 0 && nmiss <= kVictimLists && K <= 64 * nthr) {
        select_victims(m, K, nmiss);
    } else if (nmiss > 0) {
        unsigned long long myv = ~0ull;
        int mys = -1;
        for (int i = tid; i < K; i += nthr)
            if (m.lu[i] < myv) { myv = m.lu[i]; mys = i; }
        const int warp = tid >> 5, lane = tid & 31, nw = nthr >> 5;
        for (int r = 0; r < nmiss; ++r) {
            unsigned long long v = myv;
            int sl = mys;
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                unsigned long long ov = __shfl_xor_sync(0xffffffffu, v, off);
                int os = __shfl_xor_sync(0xffffffffu, sl, off);
                if (ov < v) { v = ov; sl = os; }
            }
            if (lane == 0) { m.wmin[warp] = v; m.wslot[warp] = sl; }
            __syncthreads();
            if (tid == 0) {
                unsigned long long bv = m.wmin[0];
                int bsl = m.wslot[0];
                for (int w = 1; w < nw; ++w)
                    if (m.wmin[w] < bv) { bv = m.wmin[w]; bsl = m.wslot[w]; }
                m.victims[r] = bsl;
                m.lu[bsl] = ~0ull;
            }
            __syncthreads();
            if (m.victims[r] == mys) {
                myv = ~0ull;
                mys = -1;
                for (int i = tid; i < K; i += nthr)
                    if (m.lu[i] < myv) { myv = m.lu[i]; mys = i; }
            }
        }
    }
    __syncthreads();
    // 4. assign: miss i (ascending expert) takes victim i, evicting its key
    for (int i = tid; i < nmiss; i += nthr) {
        int e = m.misses[i];
        int v = m.victims[i];
        m.u_slot[m.unit_of[e]] = v;
        if (commit) {
            int old = m.kof[v];
            if (old >= 0) c.slot_map[old] = -1;
            g_key_of[v] = layer * E + e;
            g_slot_map[e] = v;
            g_last_use[v] = clk + nh + i;
            s.copy_expert[i] = e;
            s.copy_slot[i] = v;
        }
    }
    // 5. units and their pairs
    const int n_units = nu + (c.has_shared ? 1 : 0);
    for (int u = tid; u <= n_units; u += nthr) m.u_cnt[u] = 0;
    __syncthreads();
    for (int i = tid; i < P; i += nthr) {
        int u = i < n_ids ? m.unit_of[m.ids[i]] : nu;
        m.p_unit[i] = u;
        atomicAdd(&m.u_cnt[u], 1);
    }
    __syncthreads();
    if (tid < 32) {
        // exclusive prefix over the unit counts
        int base = 0;
        for (int u0 = 0; u0 < n_units; u0 += 32) {
            int u = u0 + tid;
            int cnt = u < n_units ? m.u_cnt[u] : 0;
            int incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (tid >= off) incl += v;
            }
            if (u < n_units) m.u_cnt[u] = base + incl - cnt;
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (tid == 0) m.u_cnt[n_units] = base;
    }
    __syncthreads();
    for (int i = tid; i < P; i += nthr) {
        int u = m.p_unit[i];
        int pos = 0;
        for (int j = 0; j < i; ++j) pos += (m.p_unit[j] == u);
        if (commit) {
            s.unit_pairs[m.u_cnt[u] + pos] = i;
            s.pair_unit[i] = u;
        }
    }
    __syncthreads();
    for (int u = tid; u < n_units; u += nthr) {
        UnitDesc d;
        d.pstart = m.u_cnt[u];
        d.np = m.u_cnt[u + 1] - m.u_cnt[u];
#pragma unroll
        for (int j = 0; j < 8; ++j) d.pair8[j] = -1;
        if (u < nu) {
            const int e = m.u_expert[u];
            const int sl = m.u_slot[u];
            const uint64_t slot_addr = (uint64_t)(c.pool + ((size_t)pool * K + sl) * c.slot_stride);
            d.expert = e;
            d.slot = sl;
            d.hit = m.u_hit[u];
            if (!d.hit && c.fused_upload) {
                d.src = (uint64_t)(c.store + ((size_t)layer * E + e) * c.slot_stride);
                d.dst = slot_addr;
                if (a.spec) {
                    // predicted and prefetched one layer early: read the bank's copy
                    const int half = layer & 1;
                    const int* keys = c.bank_key + (size_t)half * c.bank_half;
                    const int nb = c.bank_n[half];
                    for (int j = 0; j < nb; ++j)
                        if (keys[j] == layer * E + e) {
                            d.src = (uint64_t)(c.bank + ((size_t)half * c.bank_half + j) * c.slot_stride);
                            if (commit) atomicAdd(c.stats + 17, 1ull);
                            break;
                        }
                }
            } else {
                d.src = slot_addr;
                d.dst = 0;
            }
            for (int j = 0; j < 3; ++j) d.g[j] = c.fmt == FMT_NVFP4 ? m.gl[e * 3 + j] : 1.0f;
        } else {
            d.expert = -1;
            d.slot = -1;
            d.hit = 1;
            d.src = (uint64_t)(c.shared_w + (size_t)layer * c.slot_stride);
            d.dst = 0;
            for (int j = 0; j < 3; ++j) d.g[j] = c.fmt == FMT_NVFP4 ? m.gl[E * 3 + j] : 1.0f;
        }
        units_out[u] = d;
        // the first eight pairs, written straight to the descriptor
        for (int i = 0, got = 0; i < P && got < 8 && got < d.np; ++i)
            if (m.p_unit[i] == u) units_out[u].pair8[got++] = i;
    }
    if (commit)
        for (int i = tid; i < n_ids; i += nthr) {
            int u = m.unit_of[m.ids[i]];
            s.slot_of[i] = m.u_slot[u];
            s.hit_of[i] = m.u_hit[u];
        }
    __syncthreads();
    if (tid == 0 && commit) {
        c.clock[pool] = clk + nu;
        Plan* pl = s.plan;
        pl->n_uniq = nu;
        pl->n_hit = nh;
        pl->n_fill = nmiss;
        pl->n_units = n_units;
        pl->status = 0;
        if (c.win) {
            c.win[2 * layer] += (unsigned)nh;
            c.win[2 * layer + 1] += (unsigned)nmiss;
        }
        unsigned long long* st = c.stats + a.bucket * 5;
        atomicAdd(st + 0, 1ull);
        atomicAdd(st + 1, (unsigned long long)nh);
        atomicAdd(st + 2, (unsigned long long)nmiss);
        atomicAdd(st + 3, (unsigned long long)nmiss * c.slot_bytes);
        if (c.trace) write_trace(c, s, layer, T, n_ids, nh, nmiss, nu);
    }
}


// Plan of a small decode call (T <= 8, so every unit has at most eight pairs)
// for a CTA that plans for itself: the same transaction as plan_decode, with
// the dedupe, the hits, the sorted misses, the assignment and the descriptors
// run by warp 0 alone, and the whole block only for the victim search. The
// unit descriptors carry their pairs in pair8 (the global pair lists are not
// written).
static __device__ __forceinline__ void plan_small(const CacheDev& c, const Scratch& s, const RouteArgs& a,
                                                  const PlanSmem& m, unsigned long long clk, const int* ids_in,
                                                  UnitDesc* units_out, bool commit) {
    const int E = c.E, k = c.k, T = a.T, layer = a.layer;
    const int n_ids = T * k;
    const int pool = c.pool_mode ? 0 : layer;
    const int K = c.K;
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int P = n_ids + (c.has_shared ? T : 0);
    const unsigned lt_mask = (1u << lane) - 1u;
    int* g_slot_map = c.slot_map + (size_t)layer * E;
    int* g_key_of = c.key_of + (size_t)pool * K;
    unsigned long long* g_last_use = c.last_use + (size_t)pool * K;
    if (warp == 0) {
        // 1. dedupe: first occurrence in [token][rank] order, numbered in that order
        for (int i = lane; i < n_ids; i += 32) {
            const int e = ids_in[i];
            m.ids[i] = e;
            atomicMin(&m.first[e], i);
        }
        __syncwarp();
        int nu = 0;
        for (int i0 = 0; i0 < n_ids; i0 += 32) {
            const int i = i0 + lane;
            const bool f = i < n_ids && m.first[m.ids[i]] == i;
            const unsigned bal = __ballot_sync(0xffffffffu, f);
            if (f) {
                const int u = nu + __popc(bal & lt_mask);
                m.unit_of[m.ids[i]] = u;
                m.u_expert[u] = m.ids[i];
            }
            nu += __popc(bal);
        }
        __syncwarp();
        // every expert of the call counts one more use (LFU)
        if (commit && c.lfu)
            for (int u = lane; u < nu; u += 32) c.uses[(size_t)layer * E + m.u_expert[u]] += 1u;
        // 2. hits, touched in unit order: stamps clock + hit rank
        int nh = 0;
        for (int u0 = 0; u0 < nu; u0 += 32) {
            const int u = u0 + lane;
            const int sl = u < nu ? m.smap[m.u_expert[u]] : -1;
            const bool h = sl >= 0;
            const unsigned bal = __ballot_sync(0xffffffffu, h);
            if (u < nu) {
                m.u_hit[u] = h;
                m.u_slot[u] = sl;
                if (h) {
                    const unsigned long long st = clk + nh + __popc(bal & lt_mask);
                    m.lu[sl] = st;
                    if (commit) g_last_use[sl] = st;
                } else {
                    atomicOr(&m.missbits[m.u_expert[u] >> 5], 1u << (m.u_expert[u] & 31));
                }
            }
            nh += __popc(bal);
        }
        __syncwarp();
        // misses in ascending expert order
        int mb = 0;
        for (int w0 = 0; w0 <= E / 32; w0 += 32) {
            const int wi = w0 + lane;
            unsigned bits = wi <= E / 32 ? m.missbits[wi] : 0u;
            const int cnt = __popc(bits);
            int incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            int pos = mb + incl - cnt;
            while (bits) {
                const int b = __ffs(bits) - 1;
                bits &= bits - 1;
                m.misses[pos++] = wi * 32 + b;
            }
            mb += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            m.scal[0] = nu;
            m.scal[1] = nh;
        }
    }
    __syncthreads();
    const int nu = m.scal[0];
    const int nh = m.scal[1];
    const int nmiss = nu - nh;
    if (c.lfu && nmiss > 0) lfu_victim_keys(c, m, clk);
    // 3. victims: the nmiss smallest stamps of the pool (LFU: keys), smallest first
    if (nmiss > 0 && nmiss <= kVictimLists && K <= 64 * nthr) {
        select_victims(m, K, nmiss);
    } else if (nmiss > 0) {
        unsigned long long myv = ~0ull;
        int mys = -1;
        for (int i = tid; i < K; i += nthr)
            if (m.lu[i] < myv) { myv = m.lu[i]; mys = i; }
        const int nw = nthr >> 5;
        for (int r = 0; r < nmiss; ++r) {
            unsigned long long v = myv;
            int sl = mys;
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                const unsigned long long ov = __shfl_xor_sync(0xffffffffu, v, off);
                const int os = __shfl_xor_sync(0xffffffffu, sl, off);
                if (ov < v) { v = ov; sl = os; }
            }
            if (lane == 0) { m.wmin[warp] = v; m.wslot[warp] = sl; }
            __syncthreads();
            if (tid == 0) {
                unsigned long long bv = m.wmin[0];
                int bsl = m.wslot[0];
                for (int w = 1; w < nw; ++w)
                    if (m.wmin[w] < bv) { bv = m.wmin[w]; bsl = m.wslot[w]; }
                m.victims[r] = bsl;
                m.lu[bsl] = ~0ull;
            }
            __syncthreads();
            if (m.victims[r] == mys) {
                myv = ~0ull;
                mys = -1;
                for (int i = tid; i < K; i += nthr)
                    if (m.lu[i] < myv) { myv = m.lu[i]; mys = i; }
            }
        }
    }
    if (warp == 0) {
        // 4. assign: miss i (ascending expert) takes victim i, evicting its key
        for (int i = lane; i < nmiss; i += 32) {
            const int e = m.misses[i];
            const int v = m.victims[i];
            m.u_slot[m.unit_of[e]] = v;
            if (commit) {
                const int old = m.kof[v];
                if (old >= 0) c.slot_map[old] = -1;
                g_key_of[v] = layer * E + e;
                g_slot_map[e] = v;
                g_last_use[v] = clk + nh + i;
                s.copy_expert[i] = e;
                s.copy_slot[i] = v;
            }
        }
        __syncwarp();
        // 5. descriptors, then each unit's pairs in ascending pair order
        const int n_units = nu + (c.has_shared ? 1 : 0);
        for (int u = lane; u < n_units; u += 32) {
            UnitDesc d;
            d.pstart = 0;
            d.np = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) d.pair8[j] = -1;
            if (u < nu) {
                const int e = m.u_expert[u];
                const int sl = m.u_slot[u];
                const uint64_t slot_addr = (uint64_t)(c.pool + ((size_t)pool * K + sl) * c.slot_stride);
                d.expert = e;
                d.slot = sl;
                d.hit = m.u_hit[u];
                if (!d.hit && c.fused_upload) {
                    d.src = (uint64_t)(c.store + ((size_t)layer * E + e) * c.slot_stride);
                    d.dst = slot_addr;
                } else {
                    d.src = slot_addr;
                    d.dst = 0;
                }
                for (int j = 0; j < 3; ++j) d.g[j] = c.fmt == FMT_NVFP4 ? m.gl[e * 3 + j] : 1.0f;
            } else {
                d.expert = -1;
                d.slot = -1;
                d.hit = 1;
                d.src = (uint64_t)(c.shared_w + (size_t)layer * c.slot_stride);
                d.dst = 0;
                for (int j = 0; j < 3; ++j) d.g[j] = c.fmt == FMT_NVFP4 ? m.gl[E * 3 + j] : 1.0f;
            }
            units_out[u] = d;
            m.u_cnt[u] = 0;
        }
        __syncwarp();
        for (int i0 = 0; i0 < P; i0 += 32) {
            const int i = i0 + lane;
            const int u = i < P ? (i < n_ids ? m.unit_of[m.ids[i]] : nu) : -1 - lane;
            const unsigned same = __match_any_sync(0xffffffffu, u);
            if (i < P) {
                const int pos = m.u_cnt[u] + __popc(same & lt_mask);
                if (pos < 8) units_out[u].pair8[pos] = i;
                __syncwarp(same);
                if (lane == 31 - __clz(same)) m.u_cnt[u] = pos + 1;
            }
            __syncwarp();
        }
        for (int u = lane; u < n_units; u += 32) units_out[u].np = m.u_cnt[u];
        if (commit) {
            for (int i = lane; i < n_ids; i += 32) {
                const int u = m.unit_of[m.ids[i]];
                s.slot_of[i] = m.u_slot[u];
                s.hit_of[i] = m.u_hit[u];
            }
            __syncwarp();
            if (lane == 0) {
                c.clock[pool] = clk + nu;
                Plan* pl = s.plan;
                pl->n_uniq = nu;
                pl->n_hit = nh;
                pl->n_fill = nmiss;
                pl->n_units = n_units;
                pl->status = 0;
                if (c.win) {
                    c.win[2 * layer] += (unsigned)nh;
                    c.win[2 * layer + 1] += (unsigned)nmiss;
                }
                unsigned long long* st = c.stats + a.bucket * 5;
                atomicAdd(st + 0, 1ull);
                atomicAdd(st + 1, (unsigned long long)nh);
                atomicAdd(st + 2, (unsigned long long)nmiss);
                atomicAdd(st + 3, (unsigned long long)nmiss * c.slot_bytes);
                if (c.trace) write_trace(c, s, layer, T, n_ids, nh, nmiss, nu);
            }
        }
    }
    __syncthreads();
}

}  // namespace moe
