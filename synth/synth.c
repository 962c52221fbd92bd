/*
 * synth.c -- seeded synthetic inputs shared by the oracle side and the CUDA
 * side: expert records in each weight format, router weights, hidden states.
 *
 * This module holds none of the MoE method's arithmetic. It only draws
 * numbers and lays them out in the canonical record formats; nothing here
 * decodes a weight or computes a layer. Every value is a pure function of
 * (seed, kind, layer, index, matrix, counter), so any expert record can be
 * produced alone, in any order and in parallel.
 *
 * Random source: a counter fed through the SplitMix64 output function
 * (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
 * OOPSLA 2014; constants as published there and in Vigna's reference code).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYN_GOLDEN 0x9E3779B97F4A7C15ULL

enum { SYN_BF16 = 0, SYN_Q4_0 = 1, SYN_FP8_B128 = 2, SYN_NVFP4 = 3 };
enum { KIND_EXPERT = 1, KIND_ROUTER = 2, KIND_HIDDEN = 3, KIND_PROMPT = 4, KIND_MISC = 5 };

uint64_t syn_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t syn_key(uint64_t seed, uint32_t kind, uint32_t a, uint32_t b, uint32_t c) {
    uint64_t k = syn_mix64(seed + SYN_GOLDEN);
    k = syn_mix64(k ^ ((uint64_t)kind << 56) ^ ((uint64_t)a << 32));
    k = syn_mix64(k ^ ((uint64_t)b << 20) ^ (uint64_t)c);
    return k;
}

static inline uint64_t rnd(uint64_t key, uint64_t ctr) { return syn_mix64(key + (ctr + 1) * SYN_GOLDEN); }

/* uniform in (0, 1] */
static inline double unif(uint64_t key, uint64_t ctr) {
    return ((double)(rnd(key, ctr) >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}

/* standard normal by Box-Muller from counters 2i and 2i+1 */
static inline double normal(uint64_t key, uint64_t i) {
    double u1 = unif(key, 2 * i), u2 = unif(key, 2 * i + 1);
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

/* round-to-nearest-even double -> bfloat16 bits (via binary32) */
static inline uint16_t to_bf16(double v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    u = u + 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static inline void put16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static inline void putf32(uint8_t* p, float f) { memcpy(p, &f, 4); } /* both hosts are little-endian */

void syn_normal_bf16(uint64_t key, size_t n, double sd, uint16_t* out) {
    size_t i;
    for (i = 0; i < n; ++i) out[i] = to_bf16(sd * normal(key, i));
}

void syn_router_weights(uint64_t seed, int layer, int E, int H, double sd, uint16_t* out) {
    syn_normal_bf16(syn_key(seed, KIND_ROUTER, (uint32_t)layer, 0, 0), (size_t)E * H, sd, out);
}

/* Prompt-style hiddens: i.i.d. N(0, sd) per (layer, token). */
void syn_prompt(uint64_t seed, int layer, int T, int H, double sd, uint16_t* out) {
    syn_normal_bf16(syn_key(seed, KIND_PROMPT, (uint32_t)layer, 0, 0), (size_t)T * H, sd, out);
}

/* Decode-style hiddens for one (layer, stream): an AR(1) sequence in fp64,
 * h_0 = e_0, h_t = rho*h_{t-1} + sqrt(1-rho^2)*e_t with e_t ~ N(0, I), each
 * step emitted as bf16. out is [nsteps][H]. */
void syn_hidden_ar1(uint64_t seed, int layer, int stream, int nsteps, int H, double rho, uint16_t* out) {
    uint64_t key = syn_key(seed, KIND_HIDDEN, (uint32_t)layer, (uint32_t)stream, 0);
    double* h = (double*)malloc(sizeof(double) * (size_t)H);
    double c = sqrt(1.0 - rho * rho);
    int t, j;
    for (t = 0; t < nsteps; ++t) {
        for (j = 0; j < H; ++j) {
            double e = normal(key, (uint64_t)t * H + j);
            h[j] = t == 0 ? e : rho * h[j] + c * e;
            out[(size_t)t * H + j] = to_bf16(h[j]);
        }
    }
    free(h);
}

/* ---- canonical record writers (layouts match the C-ABI's documentation) ---- */

static size_t mat_bytes(int fmt, int rows, int cols) {
    size_t r = (size_t)rows, c = (size_t)cols;
    switch (fmt) {
    case SYN_BF16: return r * c * 2;
    case SYN_Q4_0: return r * (c / 32) * 18;
    case SYN_FP8_B128: return r * c + ((r + 127) / 128) * ((c + 127) / 128) * 4;
    case SYN_NVFP4: return r * c / 2 + r * (c / 16);
    default: return 0;
    }
}

size_t syn_record_bytes(int fmt, int H, int I) {
    return 2 * mat_bytes(fmt, I, H) + mat_bytes(fmt, H, I) + (fmt == SYN_NVFP4 ? 12 : 0);
}

/* bf16 weights ~ N(0, 0.02). */
static void gen_bf16(uint64_t key, int rows, int cols, uint8_t* out) {
    size_t i, n = (size_t)rows * cols;
    for (i = 0; i < n; ++i) put16(out + 2 * i, to_bf16(0.02 * normal(key, i)));
}

/* Q4_0 blocks: uniform 4-bit codes; the fp16 scale is built from its bits as
 * (1 + m/1024) * 2^-9 with m uniform in 0..1023, so weights have an sd near
 * 0.013 (codes minus 8 have sd 4.6). */
static void gen_q4_0(uint64_t key, int rows, int cols, uint8_t* out) {
    size_t nblk = (size_t)rows * (cols / 32), j;
    for (j = 0; j < nblk; ++j) {
        uint8_t* blk = out + 18 * j;
        uint64_t a = rnd(key, 3 * j), b = rnd(key, 3 * j + 1);
        uint16_t m = (uint16_t)(rnd(key, 3 * j + 2) & 0x3ff);
        put16(blk, (uint16_t)((6u << 10) | m));
        memcpy(blk + 2, &a, 8);
        memcpy(blk + 10, &b, 8);
    }
}

/* FP8 e4m3 codes drawn uniformly over all bytes with the two NaN codes
 * (0x7f, 0xff) mapped to their neighbours 0x7e / 0xfe; fp32 tile scales
 * 2^-13 * (1 + U). */
static void gen_fp8(uint64_t key, int rows, int cols, uint8_t* out) {
    size_t n = (size_t)rows * cols, i;
    size_t nsc = (size_t)((rows + 127) / 128) * ((cols + 127) / 128);
    uint64_t skey = syn_mix64(key ^ 0x5ca1e5ULL);
    for (i = 0; i < n; i += 8) {
        uint64_t w = rnd(key, i / 8);
        size_t k;
        for (k = 0; k < 8 && i + k < n; ++k) {
            uint8_t b = (uint8_t)(w >> (8 * k));
            if ((b & 0x7f) == 0x7f) b = (uint8_t)(b - 1);
            out[i + k] = b;
        }
    }
    for (i = 0; i < nsc; ++i) putf32(out + n + 4 * i, (float)(ldexp(1.0, -13) * (1.0 + unif(skey, i))));
}

/* NVFP4: uniform e2m1 codes (all 16), e4m3 block scales with exponent field
 * uniform in 4..10 and any mantissa (values 2^-3 .. 15), global fp32 scale
 * 2^-9 * (1 + U) returned to the caller. */
static float gen_nvfp4(uint64_t key, int rows, int cols, uint8_t* out) {
    size_t ncode = (size_t)rows * cols / 2, nsc = (size_t)rows * (cols / 16), i;
    uint64_t skey = syn_mix64(key ^ 0x5ca1e5ULL);
    uint8_t* sc = out + ncode;
    for (i = 0; i < ncode; i += 8) {
        uint64_t w = rnd(key, i / 8);
        size_t k;
        for (k = 0; k < 8 && i + k < ncode; ++k) out[i + k] = (uint8_t)(w >> (8 * k));
    }
    for (i = 0; i < nsc; ++i) {
        uint64_t w = rnd(skey, i);
        uint8_t ex = (uint8_t)(4 + (w % 7));
        uint8_t mt = (uint8_t)((w >> 8) & 7);
        sc[i] = (uint8_t)((ex << 3) | mt);
    }
    return (float)(ldexp(1.0, -9) * (1.0 + unif(syn_mix64(key ^ 0x91063ULL), 0)));
}

/* One canonical record: gate [I x H], up [I x H], down [H x I] (+ NVFP4
 * globals). expert = -1 gives the layer's shared expert. */
int syn_expert_record(int fmt, uint64_t seed, int layer, int expert, int H, int I, uint8_t* out) {
    int m;
    uint8_t* p = out;
    float g[3];
    for (m = 0; m < 3; ++m) {
        int rows = m < 2 ? I : H, cols = m < 2 ? H : I;
        uint64_t key = syn_key(seed, KIND_EXPERT, (uint32_t)layer, (uint32_t)(expert + 1), (uint32_t)m);
        switch (fmt) {
        case SYN_BF16: gen_bf16(key, rows, cols, p); break;
        case SYN_Q4_0: gen_q4_0(key, rows, cols, p); break;
        case SYN_FP8_B128: gen_fp8(key, rows, cols, p); break;
        case SYN_NVFP4: g[m] = gen_nvfp4(key, rows, cols, p); break;
        default: return 1;
        }
        p += mat_bytes(fmt, rows, cols);
    }
    if (fmt == SYN_NVFP4) {
        putf32(p, g[0]);
        putf32(p + 4, g[1]);
        putf32(p + 8, g[2]);
    }
    return 0;
}

typedef struct {
    int fmt, layer, e0, n, H, I, stride_threads, tid;
    uint64_t seed;
    uint8_t* out;
    size_t rec;
} job_t;

static void* run_job(void* arg) {
    job_t* j = (job_t*)arg;
    int e;
    for (e = j->tid; e < j->n; e += j->stride_threads)
        syn_expert_record(j->fmt, j->seed, j->layer, j->e0 + e, j->H, j->I, j->out + (size_t)e * j->rec);
    return NULL;
}

/* Records of experts e0 .. e0+n-1 of one layer, back to back, on nthreads. */
int syn_expert_records(int fmt, uint64_t seed, int layer, int e0, int n, int H, int I, uint8_t* out,
                       int nthreads) {
    pthread_t th[64];
    job_t jobs[64];
    int t;
    size_t rec = syn_record_bytes(fmt, H, I);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 64) nthreads = 64;
    if (nthreads > n) nthreads = n > 0 ? n : 1;
    for (t = 0; t < nthreads; ++t) {
        jobs[t].fmt = fmt; jobs[t].layer = layer; jobs[t].e0 = e0; jobs[t].n = n;
        jobs[t].H = H; jobs[t].I = I; jobs[t].stride_threads = nthreads; jobs[t].tid = t;
        jobs[t].seed = seed; jobs[t].out = out; jobs[t].rec = rec;
        if (t > 0) pthread_create(&th[t], NULL, run_job, &jobs[t]);
    }
    run_job(&jobs[0]);
    for (t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    return 0;
}
