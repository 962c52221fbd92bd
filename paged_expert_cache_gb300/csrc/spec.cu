// spec.cu -- speculative next-layer routing and prefetch of expert records.
//
// "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
// experts from NVMe" (atlasrepo.com), "Workflow": run the next layer's router
// on the current layer's input and start the predicted experts' copies one
// layer early, into a second bank of GPU slots, so the loads overlap the
// current layer's compute; "Evidence": the next layer's router on the
// current layer's input picks the right top-10 65% of the time.
//
// While layer l runs, k_spec_route ranks layer l + 1's experts on layer l's
// tokens (plain fp32 logits: a prediction, not a routing decision), keeps the
// predicted experts that are not resident, and writes them to the bank half
// of layer l + 1 (layer parity), in ascending expert order; k_spec_copy then
// copies their records from the mapped host store into the bank. Layer
// l + 1's cache plan is computed exactly as without speculation; a miss whose
// record is in the bank is read from there (device memory) instead of from
// the host store, and written through to its slot as before. So speculation
// changes where a missed record's bytes come from, never the routing, the
// plan or the arithmetic.
#include "route_dev.cuh"

namespace moe {

constexpr int kSpecThreads = 256;
constexpr int kSpecWarps = kSpecThreads / 32;
constexpr int kSpecCopyCtas = 64;
constexpr uint64_t kSpecChunk = 32768;

// Logits of the next layer (one warp per expert, fp32), then the last CTA
// ranks each token, filters and fills the bank half.
__global__ void __launch_bounds__(kSpecThreads) k_spec_route(const __grid_constant__ CacheDev c,
                                                             const __grid_constant__ SpecArgs a) {
    const int E = c.E, H = c.H, k = c.k, T = a.T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kSpecWarps + warp;
    if (e < E) {
        const uint16_t* wr = a.w + (size_t)e * H;
        for (int t = 0; t < T; ++t) {
            const uint16_t* xr = a.x + (size_t)t * H;
            float acc = 0.f;
            for (int cb = lane * 8; cb < H; cb += 256) {
                const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wr + cb));
                const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xr + cb));
                const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w}, xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc = fmaf(__uint_as_float(ww[j] << 16), __uint_as_float(xx[j] << 16), acc);
                    acc = fmaf(__uint_as_float(ww[j] & 0xffff0000u), __uint_as_float(xx[j] & 0xffff0000u), acc);
                }
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) a.z[(size_t)t * E + e] = acc + (a.bias ? a.bias[e] : 0.f);
        }
    }
    __threadfence();
    __syncthreads();
    __shared__ int is_last;
    if (threadIdx.x == 0) is_last = atomicAdd(a.done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    __shared__ int pick[kSpecMaxTokens * kMaxTopK];
    __shared__ unsigned want[kMaxExperts / 32];
    for (int i = threadIdx.x; i < kMaxExperts / 32; i += blockDim.x) want[i] = 0u;
    __syncthreads();
    // warp t ranks token t: k rounds of a warp-wide maximum over the lanes'
    // best untaken experts (ties to the lower expert); the winning lane
    // looks for its next best
    if (warp < T) {
        const float* z = a.z + (size_t)warp * E;
        unsigned long long taken = 0ull;  // bit m: expert lane + 32 m is taken
        auto best_of_lane = [&]() {
            unsigned long long b = 0ull;
            for (int m = 0; lane + 32 * m < E; ++m)
                if (!((taken >> m) & 1ull)) {
                    const int ee = lane + 32 * m;
                    const unsigned long long kk =
                        ((unsigned long long)ord32(__ldcg(z + ee)) << 32) | (unsigned)(1023 - ee);
                    if (kk > b) b = kk;
                }
            return b;
        };
        unsigned long long mine = best_of_lane();
        for (int j = 0; j < k; ++j) {
            const unsigned long long best = warp_max_key(mine);
            const int ee = 1023 - (int)(best & 1023ull);
            if (lane == 0) pick[warp * k + j] = ee;
            if ((ee & 31) == lane) {
                taken |= 1ull << (ee >> 5);
                mine = best_of_lane();
            }
        }
    }
    __syncthreads();
    // predicted experts that are not resident, once each
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
        const int ee = pick[i];
        if (c.slot_map[(size_t)a.layer * E + ee] < 0) atomicOr(&want[ee >> 5], 1u << (ee & 31));
    }
    __syncthreads();
    if (warp == 0) {
        // bank slots in ascending expert order
        int n = 0;
        int* keys = c.bank_key + (size_t)a.half * c.bank_half;
        for (int w0 = 0; w0 < (E + 31) / 32; w0 += 32) {
            const int wi = w0 + lane;
            unsigned bits = wi < (E + 31) / 32 ? want[wi] : 0u;
            const int cnt = __popc(bits);
            int incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            int pos = n + incl - cnt;
            while (bits) {
                const int b = __ffs(bits) - 1;
                bits &= bits - 1;
                if (pos < c.bank_half) keys[pos] = a.layer * E + wi * 32 + b;
                ++pos;
            }
            n += __shfl_sync(0xffffffffu, incl, 31);
        }
        n = min(n, c.bank_half);
        for (int j = n + lane; j < c.bank_half; j += 32) keys[j] = -1;
        if (lane == 0) {
            c.bank_n[a.half] = n;
            atomicAdd(c.stats + 16, (unsigned long long)n);
            *a.done = 0u;
        }
    }
}

// Copies the records of the bank half's slots from the mapped host store.
__global__ void __launch_bounds__(kSpecThreads) k_spec_copy(const __grid_constant__ CacheDev c, int half) {
    const int n = c.bank_n[half];
    if (n <= 0) return;
    const uint64_t bytes = c.slot_bytes;
    const int cpr = (int)((bytes + kSpecChunk - 1) / kSpecChunk);
    const long long total = (long long)n * cpr;
    const int* keys = c.bank_key + (size_t)half * c.bank_half;
    for (long long w = blockIdx.x; w < total; w += gridDim.x) {
        const int r = (int)(w / cpr), ch = (int)(w % cpr);
        const int key = keys[r];
        const uint8_t* src = c.store + (size_t)key * c.slot_stride + (size_t)ch * kSpecChunk;
        uint8_t* dst = c.bank + ((size_t)half * c.bank_half + r) * c.slot_stride + (size_t)ch * kSpecChunk;
        const uint64_t rem = bytes - (uint64_t)ch * kSpecChunk;
        const int nv = (int)(((rem < kSpecChunk ? rem : kSpecChunk) + 15) / 16);
        for (int v0 = threadIdx.x; v0 < nv; v0 += kSpecThreads * 8) {
            uint4 buf[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int v = v0 + i * kSpecThreads;
                if (v < nv) buf[i] = ldg_stream(src + (size_t)v * 16);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int v = v0 + i * kSpecThreads;
                if (v < nv) *reinterpret_cast<uint4*>(dst + (size_t)v * 16) = buf[i];
            }
        }
    }
}

void launch_spec_route(const CacheDev& c, const SpecArgs& a, cudaStream_t st) {
    k_spec_route<<<(c.E + kSpecWarps - 1) / kSpecWarps, kSpecThreads, 0, st>>>(c, a);
}

void launch_spec_copy(const CacheDev& c, int half, cudaStream_t st) {
    k_spec_copy<<<kSpecCopyCtas, kSpecThreads, 0, st>>>(c, half);
}

}  // namespace moe
