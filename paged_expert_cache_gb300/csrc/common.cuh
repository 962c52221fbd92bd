// common.cuh -- device-side building blocks shared by the kernels of the
// routed-MoE-over-LRU-expert-cache library (sm_103a).
//
// Slot layout. A slot holds one expert's three matrices (gate, up, down) in a
// layout made for the m16n8k16 tensor-core fragment: a matrix of R rows and C
// columns is cut into 16-row tiles (rt) and 64-column chunks (kc); the bytes
// a lane needs for the four k16 steps of one (rt, kc) sit together, so one
// 16-byte load per lane feeds four MMAs. Fragment coordinates for lane l:
// g = l >> 2, q = l & 3; for k-step s the lane's A elements are
//   a0 = (row g,   cols c0+2q, c0+2q+1)    a1 = (row g+8, same cols)
//   a2 = (row g,   cols c0+2q+8, c0+2q+9)  a3 = (row g+8, same cols)
// with c0 = kc*64 + s*16 and rows relative to rt*16. Byte counts per matrix
// equal the canonical record's, so a slot is exactly a record's size.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

enum { FMT_BF16 = 0, FMT_Q4_0 = 1, FMT_FP8_B128 = 2, FMT_NVFP4 = 3 };

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 16;
constexpr int kDecodeMaxTokens = 32;

// Bytes of one matrix (R rows x C cols) in a slot; equals the canonical size.
__host__ __device__ inline uint64_t matrix_bytes(int fmt, int R, int C) {
    uint64_t r = (uint64_t)R, c = (uint64_t)C;
    switch (fmt) {
    case FMT_BF16: return r * c * 2;
    case FMT_Q4_0: return r * (c / 32) * 18;
    case FMT_FP8_B128: return r * c + ((r + 127) / 128) * ((c + 127) / 128) * 4;
    case FMT_NVFP4: return r * c / 2 + r * (c / 16);
    default: return 0;
    }
}

// Bytes between matrices inside a slot: the matrix size rounded up to 16.
__host__ __device__ inline uint64_t matrix_stride(int fmt, int R, int C) { return (matrix_bytes(fmt, R, C) + 15) & ~15ull; }

// Per-call plan, written by the routing kernel and read by the others.
struct Plan {
    int n_uniq;   // distinct routed experts of the call
    int n_hit;    // of those, resident at the start of the call
    int n_fill;   // uploads into cache slots (decode) or arena stagings (prefill)
    int n_units;  // compute units: n_uniq (+1 shared expert)
    int status;   // 0 ok; 2 capacity exceeded (nothing changed)
    int reranked; // 1 if the fp64 re-rank decided the top-k of some token
    int pool_slots;  // page-in prefill: slots the layer's pool held during the call
    int pad;
};

// One compute unit of a call (a distinct routed expert, or the shared
// expert): where its weights are read from, where a missed expert's bytes
// are written while they are read (0 for none), and its token pairs.
struct UnitDesc {
    uint64_t src;   // device address of the record the weights are read from
    uint64_t dst;   // slot the record is written into on the way (a miss), or 0
    float g[3];     // NVFP4 global scales of gate, up, down (1 otherwise)
    int pstart;     // first entry in unit_pairs
    int np;         // number of pairs
    int expert;     // routed expert id, -1 for the shared expert
    int slot;       // cache slot, -1 when staged or shared
    int hit;        // resident at the start of the call
    int pair8[8];   // the first eight entries of the unit's pair list
};
static_assert(sizeof(UnitDesc) == 80, "UnitDesc layout");

// Device pointers of one call's scratch, passed by value to kernels.
struct Scratch {
    UnitDesc* units;    // [U]
    float2* logits;     // [T][E] normalized float pair (hi, lo): hi = RN(hi + lo)
    float* bounds;      // [T][E] bound on the pair's distance from the defining fp64 sum
    int* ids;           // [T*k] rank order per token
    float* wts;         // [T*k]
    int* slot_of;       // [T*k]
    int* hit_of;        // [T*k]
    int* unit_pairs;    // [P]  pair ids: t*k + j, or T*k + t for the shared expert
    int* pair_unit;     // [P]
    uint64_t* copy_src; // [U] record copies: source (mapped host store)
    uint64_t* copy_dst; // [U] record copies: destination (slot or arena)
    int* copy_expert;   // [U] expert of each copy (the fill list)
    int* copy_slot;     // [U] slot of each copy (-1 for arena stagings)
    float* act;         // [P][I] SwiGLU activations
    float* part;        // [P][H] down-projection partials per pair
    Plan* plan;
    unsigned* route_done;   // CTA counter of the routing kernel
    unsigned* tile_done;    // [H/16] CTA counters of the down kernel
    unsigned* copy_done;    // CTA counter of the copy kernel
    unsigned long long* copy_t0;  // miss streaming start / end (globaltimer ns)
    unsigned long long* copy_t1;
    unsigned* tiles_done;   // row tiles combined by the down kernel (whole call)
    unsigned* grid_bar;     // arrival counter of the fused layer kernel's grid barriers
    unsigned* err;          // sticky device error bits (1: a grid barrier timed out, 2: a weight-slot
                            // wait timed out, 4: a prefill GEMM wait timed out)
    unsigned* logit_ctr;    // [2] logit CTAs done, per call parity (one-kernel decode)
    int2* gemm_items;       // prefill GEMM work list: (unit, 128-pair tile)
    int* gemm_count;        // its length
    int* tok_shift;         // [T] power-of-two prescale of each token row (token_shift)
    unsigned* act_amax;     // [P] largest |activation| of each pair, as fp32 bits (act_shift)
    unsigned* pass_ctr;     // [2] CTAs past the logit wait, and the call's parity (one-kernel decode)
};

// Device cache state and constants of a handle.
struct CacheDev {
    int L, E, k, H, I, fmt, has_shared, n_pools, K, norm_topk;
    int pool_mode;               // 0 per layer, 1 shared
    int fused_upload;            // 1: misses are pulled by the expert kernels themselves
    uint64_t slot_stride, slot_bytes;
    uint8_t* pool;               // [n_pools*K*stride]
    const uint8_t* store;        // mapped pinned store [L*E*stride] (device alias)
    const uint8_t* shared_w;     // [L*stride] or null
    uint8_t* arena;              // [2*group*stride] or null
    const float* gtable;         // [(L*E + L)*3] NVFP4 global scales
    int* slot_map;               // [L*E]
    int* key_of;                 // [n_pools*K]
    unsigned long long* last_use;  // [n_pools*K] clock of the last use
    unsigned long long* clock;     // [n_pools]
    unsigned* uses;                // [L*E] decode calls that routed each key (LFU)
    int lfu;                       // 1: least frequently used eviction
    unsigned long long* stats;     // [3][5], [15] re-rank count, [16] records prefetched by speculation,
                                   // [17] misses read from the prefetch bank
    uint8_t* bank;                 // speculation's prefetch bank: [2 halves][bank_half] slots, or null
    int* bank_key;                 // [2][bank_half]: layer * E + expert of each bank slot, or -1
    int* bank_n;                   // [2]: bank slots filled in each half
    int bank_half;                 // bank slots per half (layer parity)
    int pagein;                    // 1: prefill calls page their missed experts into the pool (LRU)
    // adaptive per-layer capacity (null / 0 when off): a place of a pool's
    // array holds a slot while its stamp is not ~0
    int adapt_period, adapt_step, adapt_kmin;
    int* pool_K;                   // [n_pools] slots each pool holds
    unsigned* win;                 // [L][2] hits, misses of decode calls since the last move
    unsigned long long* adapt_calls;  // decode calls so far
    unsigned long long* floor_stamp;  // [n_pools] the next stamp of an arriving slot (decreasing)
    int* trace;                    // ring of records, or null
    unsigned long long* trace_count;
    int trace_cap, trace_stride;
};

// ---------------------------------------------------------------------------
// Tensor-core helpers (mma.sync m16n8k16, fp32 accumulate).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            const void* smem_row) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(smem_row);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
    return d;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Q4_0 word -> four fp16x2 A registers holding (q - 8) exactly. Nibble pairs
// (bits 0-3|16-19) -> a0, (4-7|20-23) -> a1, (8-11|24-27) -> a2,
// (12-15|28-31) -> a3. OR-ing a nibble into the mantissa of 1024.0 gives
// 1024 + q (low position) or 1024 + 16 q (high position), both exact.
__device__ __forceinline__ void q4_to_frag(uint32_t w, uint32_t a[4]) {
    const uint32_t kMagic = 0x64006400u;  // 1024.0 in both halves
    const __half2 k1032 = u32_as_h2(0x64086408u);   // 1032.0
    const __half2 kSixteenth = u32_as_h2(0x2C002C00u);  // 1/16
    const __half2 kM72 = u32_as_h2(0xD480D480u);    // -72.0
    uint32_t t0 = lop3_and_or(w, 0x000f000fu, kMagic);
    uint32_t t1 = lop3_and_or(w, 0x00f000f0u, kMagic);
    uint32_t w8 = w >> 8;
    uint32_t t2 = lop3_and_or(w8, 0x000f000fu, kMagic);
    uint32_t t3 = lop3_and_or(w8, 0x00f000f0u, kMagic);
    a[0] = h2_as_u32(__hsub2(u32_as_h2(t0), k1032));
    a[1] = h2_as_u32(__hfma2(u32_as_h2(t1), kSixteenth, kM72));
    a[2] = h2_as_u32(__hsub2(u32_as_h2(t2), k1032));
    a[3] = h2_as_u32(__hfma2(u32_as_h2(t3), kSixteenth, kM72));
}

// Two e4m3 codes (low byte = lower column) -> fp16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two) {
    __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xffffu), __NV_E4M3);
    return (uint32_t)r.x | ((uint32_t)r.y << 16);
}

// The fp16x2 bits of two e2m1 codes (sign, 2 exponent bits, 1 mantissa bit)
// held at bits 0-3 (low half) and 16-19 (high half) of x, scaled by 2^-14:
// the code's 3 magnitude bits placed at fp16 bits 9-11 are its value's
// exponent and mantissa with fp16's bias 15 instead of e2m1's 1 (normal codes),
// or its subnormal (code 1 -> 2^-15 = 0.5 * 2^-14), and its sign goes to bit
// 15. Exact, and plain integer work: the hardware's e2m1 conversion runs on a
// pipe with a fraction of the integer rate.
__device__ __forceinline__ uint32_t e2m1x2_bits_2m14(uint32_t x) {
    return ((x << 9) & 0x0E000E00u) | ((x << 12) & 0x80008000u);
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
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
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_all;\n" ::: "memory");
}
// Closes the current group of asynchronous copies.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// Waits for every group but the most recently committed one.
__device__ __forceinline__ void cp_async_wait_but_last() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
// Asks L2 for `bytes` from `src` (16-byte aligned, a multiple of 16) without
// copying them anywhere, so later reads of them hit L2.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint2 ldg_stream8(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + expf(-v)); }

// ---------------------------------------------------------------------------
// Power-of-two prescale of the fp16 tensor-core operands.
//
// fp16 holds normal values from 2^-14 to 65504 only, while bf16 tokens reach
// about 3.4e38 and the fp32 SwiGLU activations anything fp32 holds. So each
// token row, and each pair's activation row, is multiplied by 2^-s before it
// is converted to fp16, with s chosen from the row's largest magnitude, and
// the fp32 result of its MMAs is multiplied by 2^s afterwards. Both products
// are exact (a power of two, away from fp32's overflow and subnormals), so the
// scaling changes no result except where fp16 could not hold the row:
//  - tokens: the row maximum lands at exponent 15, at most 65280 for a bf16
//    value; bf16 values down to 2^-32 of the row maximum convert exactly;
//  - activations (an fp16 hi + lo pair): the row maximum lands at exponent 14,
//    so hi never rounds up past 65504.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int prescale_shift(unsigned maxbits_f32, int top) {
    if (maxbits_f32 == 0u) return 0;
    const int e = (int)((maxbits_f32 >> 23) & 0xffu) - 127;
    const int s = e - top;
    return s < -120 ? -120 : (s > 120 ? 120 : s);
}
// 2^s as a float, for |s| <= 126.
__device__ __forceinline__ float pow2f(int s) { return __int_as_float((127 + s) << 23); }
// Shift of a token row from the largest |bf16| bit pattern of the row.
__device__ __forceinline__ int token_shift(unsigned max_abs_bf16) { return prescale_shift((max_abs_bf16 & 0x7fffu) << 16, 15); }
// Shift of an activation row from the bits of its largest |value|.
__device__ __forceinline__ int act_shift(unsigned max_abs_f32) { return prescale_shift(max_abs_f32, 14); }
// Largest |bf16| bit pattern (sign cleared) of the two halves of a word.
__device__ __forceinline__ unsigned bf16x2_absmax(uint32_t w) {
    const uint32_t m = w & 0x7fff7fffu;
    return max(m & 0xffffu, m >> 16);
}
// The SwiGLU of one (row, pair) from the unscaled-by-2^-s sums: the one
// expression every gate/up path uses, so their results agree bit for bit.
__device__ __forceinline__ float swiglu_scaled(float gs, float us, float g0, float g1, float up) {
    return silu_f(gs * g0 * up) * (us * g1 * up);
}

// Programmatic dependent launch: wait for the preceding grid's results, and
// let the following grid be scheduled.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

__device__ __forceinline__ void stg_stream(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void stg_stream8(void* p, uint2 v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};\n" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// ---------------------------------------------------------------------------
// Kernel entry points (launch helpers defined in the .cu files).
// ---------------------------------------------------------------------------
struct RouteArgs {
    const uint16_t* x;   // [T][H] bf16
    const uint16_t* w;   // [E][H] bf16
    const float* bias;   // [E] or null
    int T, layer, prefill, bucket;
    int early;           // 1: no call still in flight can write this layer's pool state, so a decode
                         // kernel may read it before waiting on the preceding grid
    int spec;            // 1: the bank half of this layer holds a speculative prefetch made for this
                         // call, complete before its expert kernels run (misses found there read it)
};

void launch_route(const CacheDev& c, const Scratch& s, const RouteArgs& a, int max_units, cudaStream_t st, bool pdl);
void launch_topk_prefill(const CacheDev& c, const Scratch& s, const RouteArgs& a, cudaStream_t st);
void launch_plan_prefill(const CacheDev& c, const Scratch& s, const RouteArgs& a, int group, cudaStream_t st);
// Page-in prefill: the cache transaction of a prefill call (after its plan),
// and the copies of the paged-in records that stay resident, from the arena
// into their slots, after the GEMMs of their staging group.
void launch_pagein(const CacheDev& c, const Scratch& s, const RouteArgs& a, cudaStream_t st);
void launch_pagein_copy(const CacheDev& c, const Scratch& s, int layer, int group, int G, cudaStream_t st);
// Adaptive per-layer capacity: after a decode call, counts it and, every
// adapt_period * L calls, moves slots between the layers' pools.
void launch_adapt(const CacheDev& c, cudaStream_t st);
void launch_copy(const CacheDev& c, const Scratch& s, int first, int count, int bucket, cudaStream_t st,
                 bool beside_compute);
void launch_gateup(const CacheDev& c, const Scratch& s, const uint16_t* x, int T, int kind, int group, int G,
                   int units, cudaStream_t st, bool pdl);
void launch_down(const CacheDev& c, const Scratch& s, float* out, int T, int kind, int group, int G, int units,
                 int bucket, cudaStream_t st, bool pdl);

// cudaLaunchKernelEx with the programmatic-serialization attribute when pdl,
// and as a cooperative launch (every CTA resident at once, or the launch is
// refused) when coop.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex_coop(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                                  bool coop, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (coop) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    if (n) {
        cfg.attrs = attr;
        cfg.numAttrs = n;
    }
    return cudaLaunchKernelEx(&cfg, k, args...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                             Args... args) {
    return launch_ex_coop(k, grid, block, smem, st, pdl, false, args...);
}
size_t route_smem_bytes(const CacheDev& c, int T);
// Fused decode layer: the dynamic shared memory a call of T tokens needs, or 0
// when the call is outside the kernel's limits; and the launch (false when
// the call does not fit, so the caller takes the three-kernel path).
size_t layer_smem_bytes(const CacheDev& c, int T);
bool launch_layer(const CacheDev& c, const Scratch& s, const RouteArgs& a, float* out, int bucket, cudaStream_t st,
                  bool pdl);
bool launch_down_rows(const CacheDev& c, const Scratch& s, float* out, int T, int units, int bucket, cudaStream_t st,
                      bool pdl);

// Prefill expert FFN as tcgen05 grouped GEMMs (gemm.cu): whether the format
// takes it, the work-list bound for P pairs over Y units, one launch over the
// units of `kind`/`group` (work list, gate/up, down), and the final combine.
bool gemm_supported(const CacheDev& c);
size_t gemm_max_items(int P, int Y);
void launch_gemm(const CacheDev& c, const Scratch& s, const uint16_t* x, int T, int kind, int group, int G, int Y,
                 cudaStream_t st);
void launch_combine(const CacheDev& c, const Scratch& s, float* out, int T, cudaStream_t st);

// Speculative next-layer routing and prefetch (spec.cu): the next layer's
// router on the current layer's tokens, its predicted non-resident experts
// written to the bank half of that layer, then their records copied there.
struct SpecArgs {
    const uint16_t* x;   // [T][H] bf16: the current layer's tokens
    const uint16_t* w;   // [E][H] bf16: the next layer's router
    const float* bias;   // [E] or null
    int T, layer, half;  // layer: the next layer; half: its bank half
    float* z;            // [T][E] fp32 logits scratch
    unsigned* done;      // CTA counter
};
constexpr int kSpecMaxTokens = 2;  // decode calls with at most this many tokens speculate
void launch_spec_route(const CacheDev& c, const SpecArgs& a, cudaStream_t st);
void launch_spec_copy(const CacheDev& c, int half, cudaStream_t st);

// Host-side repack of canonical records into the slot layout (repack.cpp).
void repack_record(int fmt, int H, int I, const uint8_t* canonical, uint8_t* slot, float* gscales3);

}  // namespace moe
