// route.cu -- router logits, top-k and the cache plan of one layer call.
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
// two-sum (a float pair whose sum carries ~48 bits), so each logit comes with
// a rigorous bound on its distance from the fp64, ascending-index sum that
// defines it. When the bound cannot separate the ranking, the candidates are
// recomputed exactly in that definition's order (sequential fp64, no fused
// multiply-add) and ranked again.
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

// Logits of one CTA's experts for one CTA's tokens. Writes logits (double)
// and bounds (double) per (token, expert).
__device__ void router_logits_tile(const CacheDev& c, const Scratch& s, const RouteArgs& a, uint8_t* smem,
                                   double* logits, double* bounds) {
    const int H = c.H, E = c.E;
    const int t0 = blockIdx.y * kRouteTokens;
    const int nt = min(kRouteTokens, a.T - t0);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);  // [kRouteTokens][H]
    const int vec_per_row = H / 8;
    for (int i = threadIdx.x; i < nt * vec_per_row; i += blockDim.x) {
        int tt = i / vec_per_row, cv = i - tt * vec_per_row;
        reinterpret_cast<uint4*>(xs + (size_t)tt * H)[cv] =
            reinterpret_cast<const uint4*>(a.x + (size_t)(t0 + tt) * H)[cv];
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kRouteWarps + warp;
    if (e >= E) return;
    float hi[kRouteTokens], lo[kRouteTokens], ab[kRouteTokens];
#pragma unroll
    for (int tt = 0; tt < kRouteTokens; ++tt) hi[tt] = lo[tt] = ab[tt] = 0.f;
    const uint16_t* wr = a.w + (size_t)e * H;
    for (int cb = lane * 8; cb < H; cb += 256) {
        uint4 wv = *reinterpret_cast<const uint4*>(wr + cb);
        float wf[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                       bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
#pragma unroll
        for (int tt = 0; tt < kRouteTokens; ++tt) {
            if (tt < nt) {
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
        for (int tt = 0; tt < kRouteTokens; ++tt) {
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
    if (lane == 0) {
        // Bound: the float-pair sum is within g^2 * S of the exact sum (g =
        // n u / (1 - n u), n the longest chain of roundings, u = 2^-24), the
        // fp64 definition is within 2048*2^-53 * S plus its bias rounding, and
        // forming the double costs 2^-53 |z|. Doubled for margin.
        const double n = (double)(H / 32 + 16);
        const double g = n * 0x1p-24 / (1.0 - n * 0x1p-24);
        const double sbound = 0x1p-52 * (double)H;
        for (int tt = 0; tt < nt; ++tt) {
            double S = (double)ab[tt] * (1.0 + 2.0 * g);
            double z = (double)hi[tt] + (double)lo[tt];
            if (a.bias) z = z + (double)a.bias[e];
            double beta = 2.0 * (g * g * S + sbound * S + 0x1p-50 * fabs(z)) + (double)H * 0x1p-148 + 1e-300;
            logits[(size_t)(t0 + tt) * E + e] = z;
            bounds[(size_t)(t0 + tt) * E + e] = beta;
        }
    }
}

// The logit of (t, e) exactly as the definition states it: fp64, ascending
// h, a product then an add at every step, then the bias.
__device__ double exact_logit(const RouteArgs& a, int H, int t, int e) {
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

// Warp-wide argmax by (value desc, index asc) over per-lane candidates.
__device__ __forceinline__ void warp_best(double& z, int& e) {
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        double oz = __shfl_xor_sync(0xffffffffu, z, off);
        int oe = __shfl_xor_sync(0xffffffffu, e, off);
        if (better(oz, oe, z, e)) { z = oz; e = oe; }
    }
}

// Top-k of token t by one warp. zs/bs: per-warp smem of E doubles each,
// cand: per-warp smem of E ints.
__device__ void topk_token(const CacheDev& c, const Scratch& s, const RouteArgs& a, const double* logits,
                           const double* bounds, int t, double* zs, double* bs, int* cand,
                           unsigned long long* rerank_flag) {
    const int E = c.E, k = c.k, lane = threadIdx.x & 31;
    for (int e = lane; e < E; e += 32) {
        zs[e] = __ldcg(logits + (size_t)t * E + e);
        bs[e] = __ldcg(bounds + (size_t)t * E + e);
    }
    __syncwarp();
    // k rounds of argmax over the untaken experts; bit m of `taken` is e = lane + 32 m
    unsigned taken = 0;
    int sel[kMaxTopK];
    double selz[kMaxTopK];
    for (int j = 0; j < k; ++j) {
        double bz = -INFINITY;
        int be = 0x7fffffff;
        for (int e = lane, m = 0; e < E; e += 32, ++m)
            if (!((taken >> m) & 1u) && better(zs[e], e, bz, be)) { bz = zs[e]; be = e; }
        warp_best(bz, be);
        sel[j] = be;
        selz[j] = bz;
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
    }
    // max upper bound over the experts not picked
    double mx = -INFINITY;
    for (int e = lane, m = 0; e < E; e += 32, ++m)
        if (!((taken >> m) & 1u)) mx = fmax(mx, zs[e] + bs[e]);
#pragma unroll
    for (int off = 16; off; off >>= 1) mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    // certify: each pick's lower bound is above every later upper bound
    bool ok = true;
    double run = mx, lam = INFINITY;
    for (int j = k - 1; j >= 0; --j) {
        double zj = selz[j], bj = bs[sel[j]];
        if (!(zj - bj > run)) ok = false;
        run = fmax(run, zj + bj);
        lam = fmin(lam, zj - bj);
    }
    int ids[kMaxTopK];
    double idz[kMaxTopK];
    for (int j = 0; j < k; ++j) { ids[j] = sel[j]; idz[j] = selz[j]; }
    if (!ok) {
        // candidates: every expert whose upper bound reaches the lowest lower
        // bound of the picks; outside this set no expert can be in the top-k
        int nc = 0;
        for (int base = 0; base < E; base += 32) {
            int e = base + lane;
            bool in = e < E && zs[e] + bs[e] >= lam;
            unsigned bal = __ballot_sync(0xffffffffu, in);
            if (in) cand[nc + __popc(bal & ((1u << lane) - 1u))] = e;
            nc += __popc(bal);
        }
        __syncwarp();
        for (int i = lane; i < nc; i += 32) zs[cand[i]] = exact_logit(a, c.H, t, cand[i]);
        __syncwarp();
        // k rounds over the candidates; a picked candidate is marked by
        // storing -1 - e in its cand entry
        for (int j = 0; j < k; ++j) {
            double bz = -INFINITY;
            int be = 0x7fffffff, bi = -1;
            for (int i = lane; i < nc; i += 32) {
                int e = cand[i];
                if (e >= 0 && better(zs[e], e, bz, be)) { bz = zs[e]; be = e; bi = i; }
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                double oz = __shfl_xor_sync(0xffffffffu, bz, off);
                int oe = __shfl_xor_sync(0xffffffffu, be, off);
                int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (better(oz, oe, bz, be)) { bz = oz; be = oe; bi = oi; }
            }
            ids[j] = be;
            idz[j] = bz;
            if (lane == (bi & 31)) cand[bi] = -1 - be;
            __syncwarp();
        }
        if (lane == 0) atomicExch(rerank_flag, 1ull);
    }
    // combine weights in fp32 from the picks' logits
    if (lane == 0) {
        float w[kMaxTopK];
        float sum = 0.f;
        if (c.norm_topk) {
            for (int j = 0; j < k; ++j) { w[j] = expf((float)(idz[j] - idz[0])); sum += w[j]; }
        } else {
            double zmax = -INFINITY;
            for (int e = 0; e < E; ++e) zmax = fmax(zmax, zs[e]);
            for (int e = 0; e < E; ++e) sum += expf((float)(zs[e] - zmax));
            for (int j = 0; j < k; ++j) w[j] = expf((float)(idz[j] - zmax));
        }
        for (int j = 0; j < k; ++j) {
            s.ids[t * k + j] = ids[j];
            s.wts[t * k + j] = w[j] / sum;
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// Plan of a decode call (T <= 32): the cache transaction, run by one CTA.
// ---------------------------------------------------------------------------
struct PlanSmem {
    int* first;       // [E] first pair index routed to e (or INT_MAX)
    int* unit_of;     // [E]
    unsigned* missbits;  // [E/32 + 1]
    int* u_expert;    // [U]
    int* u_slot;      // [U]
    int* u_hit;       // [U]
    int* u_cnt;       // [U+1]
    int* p_unit;      // [P]
    unsigned long long* lu;  // [K] last-use stamps of the pool
    unsigned long long* wmin;  // [8]
    int* wslot;       // [8]
    int* victims;     // [U]
    int* misses;      // [U] miss experts ascending
    int* scal;        // [8]: 0 n_uniq, 1 n_hit, 2 n_miss
};

__device__ void write_trace(const CacheDev& c, const Scratch& s, int layer, int T, int n_ids, int n_hit,
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

__device__ void plan_decode(const CacheDev& c, const Scratch& s, const RouteArgs& a, uint8_t* smem) {
    const int E = c.E, k = c.k, T = a.T, layer = a.layer;
    const int n_ids = T * k;
    const int pool = c.pool_mode ? 0 : layer;
    const int K = c.K;
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int U = min(n_ids, E) + 1;
    const int P = n_ids + (c.has_shared ? T : 0);
    PlanSmem m;
    uint8_t* p = smem;
    auto take = [&](size_t bytes) { uint8_t* q = p; p += (bytes + 15) & ~(size_t)15; return q; };
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
    m.wmin = (unsigned long long*)take(sizeof(unsigned long long) * 32);
    m.wslot = (int*)take(sizeof(int) * 32);
    m.scal = (int*)take(sizeof(int) * 8);
    m.lu = (unsigned long long*)take(sizeof(unsigned long long) * K);

    int* slot_map = c.slot_map + (size_t)layer * E;
    int* key_of = c.key_of + (size_t)pool * K;
    unsigned long long* last_use = c.last_use + (size_t)pool * K;

    // 1. dedupe: first occurrence in [token][rank] order
    for (int e = tid; e < E; e += nthr) m.first[e] = 0x7fffffff;
    for (int i = tid; i <= E / 32; i += nthr) m.missbits[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n_ids; i += nthr) atomicMin(&m.first[s.ids[i]], i);
    __syncthreads();
    if (tid < 32) {
        // unit index = rank of the first occurrence among first occurrences
        int base = 0;
        for (int i0 = 0; i0 < n_ids; i0 += 32) {
            int i = i0 + tid;
            bool f = i < n_ids && m.first[s.ids[i]] == i;
            unsigned bal = __ballot_sync(0xffffffffu, f);
            if (f) {
                int u = base + __popc(bal & ((1u << tid) - 1u));
                m.unit_of[s.ids[i]] = u;
                m.u_expert[u] = s.ids[i];
            }
            base += __popc(bal);
        }
        if (tid == 0) m.scal[0] = base;
    }
    __syncthreads();
    const int nu = m.scal[0];
    // 2. hits: touched in unit order, stamps clock + hit rank
    const unsigned long long clk = c.clock[pool];
    if (tid < 32) {
        int base = 0;
        for (int u0 = 0; u0 < nu; u0 += 32) {
            int u = u0 + tid;
            int sl = u < nu ? slot_map[m.u_expert[u]] : -1;
            bool h = sl >= 0;
            unsigned bal = __ballot_sync(0xffffffffu, h);
            if (u < nu) {
                m.u_hit[u] = h;
                m.u_slot[u] = sl;
                if (h) last_use[sl] = clk + base + __popc(bal & ((1u << tid) - 1u));
                else atomicOr(&m.missbits[m.u_expert[u] >> 5], 1u << (m.u_expert[u] & 31));
            }
            base += __popc(bal);
        }
        if (tid == 0) m.scal[1] = base;
    }
    __syncthreads();
    const int nh = m.scal[1];
    const int nmiss = nu - nh;
    // misses in ascending expert order
    if (tid < 32) {
        int base = 0;
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
            int pos = base + incl - cnt;
            while (bits) {
                int b = __ffs(bits) - 1;
                bits &= bits - 1;
                m.misses[pos++] = wi * 32 + b;
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    // 3. victims: the nmiss smallest stamps of the pool, smallest first
    for (int i = tid; i < K; i += nthr) m.lu[i] = last_use[i];
    __syncthreads();
    if (nmiss > 0) {
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
            int taken = m.victims[r];
            if (taken == mys) {
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
        int old = key_of[v];
        if (old >= 0) c.slot_map[old] = -1;
        key_of[v] = layer * E + e;
        slot_map[e] = v;
        last_use[v] = clk + nh + i;
        m.u_slot[m.unit_of[e]] = v;
        s.copy_expert[i] = e;
        s.copy_slot[i] = v;
        s.copy_src[i] = (uint64_t)(c.store + ((size_t)layer * E + e) * c.slot_stride);
        s.copy_dst[i] = (uint64_t)(c.pool + ((size_t)pool * K + v) * c.slot_stride);
    }
    __syncthreads();
    // 5. units and pairs
    const int n_units = nu + (c.has_shared ? 1 : 0);
    for (int u = tid; u <= n_units; u += nthr) m.u_cnt[u] = 0;
    __syncthreads();
    for (int i = tid; i < P; i += nthr) {
        int u = i < n_ids ? m.unit_of[s.ids[i]] : nu;
        m.p_unit[i] = u;
        atomicAdd(&m.u_cnt[u], 1);
    }
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int u = 0; u < n_units; ++u) {
            int cnt = m.u_cnt[u];
            s.unit_pstart[u] = acc;
            m.u_cnt[u] = acc;
            acc += cnt;
        }
        s.unit_pstart[n_units] = acc;
    }
    __syncthreads();
    for (int i = tid; i < P; i += nthr) {
        int u = m.p_unit[i];
        int pos = 0;
        for (int j = 0; j < i; ++j) pos += (m.p_unit[j] == u);
        s.unit_pairs[m.u_cnt[u] + pos] = i;
        s.pair_unit[i] = u;
    }
    for (int u = tid; u < n_units; u += nthr) {
        if (u < nu) {
            int e = m.u_expert[u];
            s.unit_expert[u] = e;
            s.unit_slot[u] = m.u_slot[u];
            s.unit_src[u] = (uint64_t)(c.pool + ((size_t)pool * K + m.u_slot[u]) * c.slot_stride);
            for (int j = 0; j < 3; ++j) s.unit_g[u * 3 + j] = c.gtable[((size_t)layer * E + e) * 3 + j];
        } else {
            s.unit_expert[u] = -1;
            s.unit_slot[u] = -1;
            s.unit_src[u] = (uint64_t)(c.shared_w + (size_t)layer * c.slot_stride);
            for (int j = 0; j < 3; ++j) s.unit_g[u * 3 + j] = c.gtable[((size_t)c.L * E + layer) * 3 + j];
        }
    }
    for (int i = tid; i < n_ids; i += nthr) {
        int u = m.unit_of[s.ids[i]];
        s.slot_of[i] = m.u_slot[u];
        s.hit_of[i] = m.u_hit[u];
    }
    __syncthreads();
    if (tid == 0) {
        c.clock[pool] = clk + nu;
        Plan* pl = s.plan;
        pl->n_uniq = nu;
        pl->n_hit = nh;
        pl->n_fill = nmiss;
        pl->n_units = n_units;
        pl->status = 0;
        unsigned long long* st = c.stats + a.bucket * 5;
        st[0] += 1;
        st[1] += (unsigned long long)nh;
        st[2] += (unsigned long long)nmiss;
        st[3] += (unsigned long long)nmiss * c.slot_bytes;
        if (c.trace) write_trace(c, s, layer, T, n_ids, nh, nmiss, nu);
    }
}

// Fused decode routing: all CTAs compute logits; the last CTA to finish
// ranks every token and runs the plan.
__global__ void __launch_bounds__(kRouteThreads) k_route(CacheDev c, Scratch s, RouteArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    double* logits = s.logits;
    double* bounds = s.bounds;
    router_logits_tile(c, s, a, smem, logits, bounds);
    if (a.prefill) return;
    __threadfence();
    __syncthreads();
    __shared__ int is_last;
    if (threadIdx.x == 0) {
        unsigned total = gridDim.x * gridDim.y;
        is_last = atomicAdd(s.route_done, 1u) == total - 1;
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    const int warp = threadIdx.x >> 5;
    const int E = c.E;
    __shared__ unsigned long long rerank;
    if (threadIdx.x == 0) rerank = 0;
    __syncthreads();
    double* zs = reinterpret_cast<double*>(smem) + (size_t)warp * 2 * E;
    double* bs = zs + E;
    int* cand = reinterpret_cast<int*>(reinterpret_cast<double*>(smem) + (size_t)kRouteWarps * 2 * E) + warp * E;
    for (int t = warp; t < a.T; t += kRouteWarps) topk_token(c, s, a, logits, bounds, t, zs, bs, cand, &rerank);
    __syncthreads();
    if (threadIdx.x == 0) {
        *s.route_done = 0;
        if (rerank) { c.stats[15] += 1; s.plan->reranked = 1; } else s.plan->reranked = 0;
    }
    __syncthreads();
    plan_decode(c, s, a, smem);
}

// Prefill: one warp per token.
__global__ void __launch_bounds__(kRouteThreads) k_topk(CacheDev c, Scratch s, RouteArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, E = c.E;
    const int t = blockIdx.x * kRouteWarps + warp;
    __shared__ unsigned long long rerank;
    if (threadIdx.x == 0) rerank = 0;
    __syncthreads();
    double* zs = reinterpret_cast<double*>(smem) + (size_t)warp * 2 * E;
    double* bs = zs + E;
    int* cand = reinterpret_cast<int*>(reinterpret_cast<double*>(smem) + (size_t)kRouteWarps * 2 * E) + warp * E;
    if (t < a.T)
        topk_token(c, s, a, s.logits, s.bounds, t, zs, bs,
                   cand, &rerank);
    __syncthreads();
    if (threadIdx.x == 0 && rerank) atomicAdd(c.stats + 15, 1ull);
}

// Prefill plan: read-only lookup. Units: resident experts ascending, then
// staged experts ascending (so groups of `group` are contiguous ranges).
__global__ void __launch_bounds__(1024) k_plan_prefill(CacheDev c, Scratch s, RouteArgs a, int group) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int E = c.E, k = c.k, T = a.T, layer = a.layer;
    const int n_ids = T * k;
    const int P = n_ids + (c.has_shared ? T : 0);
    const int tid = threadIdx.x, nthr = blockDim.x;
    int* used = reinterpret_cast<int*>(smem);  // [E]
    int* unit_of = used + E;                   // [E]
    int* cnt = unit_of + E;                    // [E+1]
    int* cur = cnt + E + 1;                    // [E+1]
    __shared__ int nh_s, nu_s;
    int* slot_map = c.slot_map + (size_t)layer * E;
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
    for (int e = tid; e < E; e += nthr) {
        if (!used[e]) continue;
        int u = unit_of[e];
        bool hit = slot_map[e] >= 0;
        s.unit_expert[u] = e;
        s.unit_slot[u] = hit ? slot_map[e] : -1;
        int pool = c.pool_mode ? 0 : layer;
        s.unit_src[u] = hit ? (uint64_t)(c.pool + ((size_t)pool * c.K + slot_map[e]) * c.slot_stride)
                            : s.copy_dst[u - nh];
        for (int j = 0; j < 3; ++j) s.unit_g[u * 3 + j] = c.gtable[((size_t)layer * E + e) * 3 + j];
    }
    if (tid == 0 && c.has_shared) {
        s.unit_expert[nu] = -1;
        s.unit_slot[nu] = -1;
        s.unit_src[nu] = (uint64_t)(c.shared_w + (size_t)layer * c.slot_stride);
        for (int j = 0; j < 3; ++j) s.unit_g[nu * 3 + j] = c.gtable[((size_t)c.L * E + layer) * 3 + j];
    }
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
            s.unit_pstart[u] = acc;
            cur[u] = acc;
            acc += cnt[u];
        }
        s.unit_pstart[n_units] = acc;
    }
    __syncthreads();
    for (int i = tid; i < P; i += nthr) {
        int u = s.pair_unit[i];
        s.unit_pairs[atomicAdd(&cur[u], 1)] = i;
    }
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
        unsigned long long* st = c.stats + a.bucket * 5;
        st[0] += 1;
        st[1] += (unsigned long long)nh;
        st[2] += (unsigned long long)(nu - nh);
        st[3] += (unsigned long long)(nu - nh) * c.slot_bytes;
        if (c.trace) write_trace(c, s, layer, T, n_ids, nh, nu - nh, nu);
    }
}

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------
static size_t topk_smem(int E) { return (size_t)kRouteWarps * E * (2 * sizeof(double) + sizeof(int)); }

static size_t plan_smem(const CacheDev& c, int T) {
    int n_ids = T * c.k;
    int U = min(n_ids, c.E) + 1;
    int P = n_ids + (c.has_shared ? T : 0);
    size_t b = 0;
    auto add = [&](size_t x) { b += (x + 15) & ~(size_t)15; };
    add(sizeof(int) * c.E);
    add(sizeof(int) * c.E);
    add(sizeof(unsigned) * (c.E / 32 + 1));
    for (int i = 0; i < 4; ++i) add(sizeof(int) * (U + 1));
    add(sizeof(int) * P);
    add(sizeof(int) * U);
    add(sizeof(int) * U);
    add(sizeof(unsigned long long) * 32);
    add(sizeof(int) * 32);
    add(sizeof(int) * 8);
    add(sizeof(unsigned long long) * c.K);
    return b;
}

size_t route_smem_bytes(const CacheDev& c, int T) {
    size_t x = (size_t)kRouteTokens * c.H * sizeof(uint16_t);
    size_t tk = topk_smem(c.E);
    size_t pl = plan_smem(c, T);
    size_t m = x > tk ? x : tk;
    return m > pl ? m : pl;
}

void launch_route(const CacheDev& c, const Scratch& s, const RouteArgs& a, int /*max_units*/, cudaStream_t st) {
    dim3 grid((c.E + kRouteWarps - 1) / kRouteWarps, (a.T + kRouteTokens - 1) / kRouteTokens);
    size_t sm = a.prefill ? (size_t)kRouteTokens * c.H * sizeof(uint16_t) : route_smem_bytes(c, a.T);
    static size_t set_route = 0;
    if (sm > set_route) {
        cudaFuncSetAttribute(k_route, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        set_route = sm;
    }
    k_route<<<grid, kRouteThreads, sm, st>>>(c, s, a);
}

void launch_topk_prefill(const CacheDev& c, const Scratch& s, const RouteArgs& a, cudaStream_t st) {
    size_t sm = topk_smem(c.E);
    static size_t set_topk = 0;
    if (sm > set_topk) {
        cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        set_topk = sm;
    }
    k_topk<<<(a.T + kRouteWarps - 1) / kRouteWarps, kRouteThreads, sm, st>>>(c, s, a);
}

void launch_plan_prefill(const CacheDev& c, const Scratch& s, const RouteArgs& a, int group, cudaStream_t st) {
    size_t sm = sizeof(int) * (4 * (size_t)c.E + 2);
    static size_t set_plan = 0;
    if (sm > set_plan) {
        cudaFuncSetAttribute(k_plan_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        set_plan = sm;
    }
    k_plan_prefill<<<1, 1024, sm, st>>>(c, s, a, group);
}

}  // namespace moe
