/*
 * moe_oracle.c -- CPU oracle for the routed MoE FFN over an LRU expert cache.
 *
 * TEST INFRASTRUCTURE (see moe_oracle.h): the slow reference the CUDA path is
 * checked against. Only tests, the smoke check and the benchmark's CPU
 * baseline may load it; the product never does.
 *
 * Everything is fp64 and single threaded. Build with -ffp-contract=off.
 * Page tags ([EXPLAINER], [PAGED], [T4], [FP4LOCAL], [NVME]) are defined in
 * moe_oracle.h with the pages' titles.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Scalar decoders                                                           */
/* ------------------------------------------------------------------------ */

/* IEEE-754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.
 * The Q4_0 block scale is this 2-byte type [EXPLAINER, "The bus problem"]. */
double orc_decode_fp16(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24); /* subnormal: frac/1024 * 2^-14 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp(1.0 + (double)frac / 1024.0, expo - 15);
    }
    return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double orc_decode_bf16(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 7) & 0xff;
    int frac = bits & 0x7f;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -133); /* subnormal: frac/128 * 2^-126 */
    } else if (expo == 255) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp(1.0 + (double)frac / 128.0, expo - 127);
    }
    return sign ? -v : v;
}

/* OCP FP8 E4M3 ("FN" variant): 1 sign, 4 exponent (bias 7), 3 fraction
 * bits; exponent field 0 is subnormal (frac/8 * 2^-6); there are no
 * infinities and only S.1111.111 is NaN, so the largest value is 448. */
double orc_decode_e4m3(uint8_t bits) {
    int sign = (bits >> 7) & 1;
    int expo = (bits >> 3) & 0xf;
    int frac = bits & 0x7;
    double v;
    if (expo == 15 && frac == 7) return NAN;
    if (expo == 0) {
        v = ldexp((double)frac, -9);
    } else {
        v = ldexp(1.0 + (double)frac / 8.0, expo - 7);
    }
    return sign ? -v : v;
}

/* OCP FP4 E2M1: 1 sign (bit 3), 2 exponent (bias 1), 1 fraction bit;
 * exponent field 0 is subnormal (frac * 0.5). Magnitudes 0, .5, 1, 1.5, 2,
 * 3, 4, 6; no infinities or NaN. */
double orc_decode_e2m1(uint8_t nibble) {
    int sign = (nibble >> 3) & 1;
    int expo = (nibble >> 1) & 0x3;
    int frac = nibble & 0x1;
    double v;
    if (expo == 0) {
        v = 0.5 * (double)frac;
    } else {
        v = ldexp(1.0 + (double)frac / 2.0, expo - 1);
    }
    return sign ? -v : v;
}

int orc_decode_array(int kind, const void* in, size_t n, double* out) {
    size_t i;
    if (kind == 0 || kind == 1) {
        const uint8_t* p = (const uint8_t*)in;
        for (i = 0; i < n; ++i) {
            uint16_t b = (uint16_t)(p[2 * i] | (p[2 * i + 1] << 8));
            out[i] = kind == 0 ? orc_decode_fp16(b) : orc_decode_bf16(b);
        }
        return ORC_OK;
    }
    if (kind == 2 || kind == 3) {
        const uint8_t* p = (const uint8_t*)in;
        for (i = 0; i < n; ++i) out[i] = kind == 2 ? orc_decode_e4m3(p[i]) : orc_decode_e2m1(p[i]);
        return ORC_OK;
    }
    return ORC_ERR_INVALID;
}

/* Lookup tables filled by calling the decoders above once; a table entry is
 * by construction the decoder's value for that code. */
static double g_e4m3[256];
static double g_e2m1[16];
static int g_tables_ready = 0;

static void build_tables(void) {
    int i;
    if (g_tables_ready) return;
    for (i = 0; i < 256; ++i) g_e4m3[i] = orc_decode_e4m3((uint8_t)i);
    for (i = 0; i < 16; ++i) g_e2m1[i] = orc_decode_e2m1((uint8_t)i);
    g_tables_ready = 1;
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

static double rdf32(const uint8_t* p) {
    uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Record geometry                                                           */
/* ------------------------------------------------------------------------ */

/* Q4_0: blocks of 32 consecutive weights of a row, each an fp16 scale then
 * 16 bytes of codes: 18 bytes per 32 weights [EXPLAINER, "The bus problem"].
 * FP8_B128: e4m3 codes row-major, then fp32 scales over 128x128 tiles.
 * NVFP4: e2m1 codes two per byte, then one e4m3 scale per 16 weights of a
 * row; the fp32 global scale of each matrix sits at the end of the record. */
size_t orc_matrix_bytes(int fmt, int rows, int cols) {
    size_t r = (size_t)rows, c = (size_t)cols;
    switch (fmt) {
    case ORC_FMT_BF16: return r * c * 2;
    case ORC_FMT_Q4_0: return (cols % 32) ? 0 : r * (c / 32) * 18;
    case ORC_FMT_FP8_B128: return r * c + ((r + 127) / 128) * ((c + 127) / 128) * 4;
    case ORC_FMT_NVFP4: return (cols % 16) ? 0 : r * c / 2 + r * (c / 16);
    default: return 0;
    }
}

size_t orc_slot_bytes(int fmt, int H, int I) {
    return 2 * orc_matrix_bytes(fmt, I, H) + orc_matrix_bytes(fmt, H, I);
}

size_t orc_record_bytes(int fmt, int H, int I) {
    return orc_slot_bytes(fmt, H, I) + (fmt == ORC_FMT_NVFP4 ? 12 : 0);
}

int64_t orc_slots_for_budget(double pool_bytes, double slot_bytes) {
    if (slot_bytes <= 0) return 0;
    return (int64_t)floor(pool_bytes / slot_bytes);
}

/* Dequantise row r of a canonical matrix into w[cols]. */
static void dequant_row(int fmt, const uint8_t* mat, int rows, int cols, double g, int r, double* w) {
    int c, b, i;
    build_tables();
    if (fmt == ORC_FMT_BF16) {
        const uint8_t* row = mat + (size_t)r * cols * 2;
        for (c = 0; c < cols; ++c) w[c] = orc_decode_bf16(rd16(row + 2 * c));
    } else if (fmt == ORC_FMT_Q4_0) {
        /* w = d * (q - 8); byte i of a block holds element i in its low
         * nibble and element i + 16 in its high nibble. */
        int nb = cols / 32;
        const uint8_t* row = mat + (size_t)r * nb * 18;
        for (b = 0; b < nb; ++b) {
            const uint8_t* blk = row + (size_t)b * 18;
            double d = orc_decode_fp16(rd16(blk));
            for (i = 0; i < 16; ++i) {
                int lo = blk[2 + i] & 0x0f;
                int hi = blk[2 + i] >> 4;
                w[32 * b + i] = d * (double)(lo - 8);
                w[32 * b + 16 + i] = d * (double)(hi - 8);
            }
        }
    } else if (fmt == ORC_FMT_FP8_B128) {
        /* w[r,c] = e4m3(q[r,c]) * s[r/128, c/128] */
        const uint8_t* row = mat + (size_t)r * cols;
        const uint8_t* scales = mat + (size_t)rows * cols;
        int ncb = (cols + 127) / 128;
        for (c = 0; c < cols; ++c) {
            double s = rdf32(scales + 4 * ((size_t)(r / 128) * ncb + (size_t)(c / 128)));
            w[c] = g_e4m3[row[c]] * s;
        }
    } else if (fmt == ORC_FMT_NVFP4) {
        /* w = e2m1(q) * e4m3(s_block16) * g; low nibble = even element. */
        const uint8_t* row = mat + (size_t)r * (cols / 2);
        const uint8_t* scales = mat + (size_t)rows * (cols / 2) + (size_t)r * (cols / 16);
        for (c = 0; c < cols; ++c) {
            uint8_t byte = row[c / 2];
            uint8_t nib = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0x0f);
            w[c] = g_e2m1[nib] * g_e4m3[scales[c / 16]] * g;
        }
    }
}

int orc_dequant_matrix(int fmt, const uint8_t* mat, int rows, int cols, double g, double* out) {
    int r;
    if (orc_matrix_bytes(fmt, rows, cols) == 0) return ORC_ERR_INVALID;
    for (r = 0; r < rows; ++r) dequant_row(fmt, mat, rows, cols, g, r, out + (size_t)r * cols);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Router: logits, top-k, weights                                            */
/* ------------------------------------------------------------------------ */

/* The router scores every expert for each token and keeps a few [EXPLAINER,
 * "The model that should not fit"]: one logit per expert, a plain dot
 * product summed in ascending h, then the per-expert bias. */
void orc_router_logits(const uint16_t* x_bf16, int T, int H, const uint16_t* w_bf16, int E,
                       const float* bias, double* z) {
    int t, e, h;
    for (t = 0; t < T; ++t) {
        for (e = 0; e < E; ++e) {
            double acc = 0.0;
            for (h = 0; h < H; ++h) {
                double prod = orc_decode_bf16(x_bf16[(size_t)t * H + h]) *
                              orc_decode_bf16(w_bf16[(size_t)e * H + h]);
                acc = acc + prod;
            }
            if (bias) acc = acc + (double)bias[e];
            z[(size_t)t * E + e] = acc;
        }
    }
}

/* k largest logits per token, in rank order; equal logits go to the lower
 * expert id (a later expert must be strictly larger to displace it). */
void orc_topk(const double* z, int T, int E, int k, int norm, int32_t* ids, double* wts) {
    int t, j, e;
    char* taken = (char*)calloc((size_t)E, 1);
    for (t = 0; t < T; ++t) {
        const double* zt = z + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (j = 0; j < k; ++j) {
            int best = -1;
            for (e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || zt[e] > zt[best]) best = e;
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        if (norm) {
            /* softmax restricted to the selected logits */
            double zmax = zt[ids[(size_t)t * k]];
            double sum = 0.0;
            for (j = 0; j < k; ++j) sum += exp(zt[ids[(size_t)t * k + j]] - zmax);
            for (j = 0; j < k; ++j) wts[(size_t)t * k + j] = exp(zt[ids[(size_t)t * k + j]] - zmax) / sum;
        } else {
            /* full softmax over all E, read at the selected experts */
            double zmax = zt[0], sum = 0.0;
            for (e = 1; e < E; ++e)
                if (zt[e] > zmax) zmax = zt[e];
            for (e = 0; e < E; ++e) sum += exp(zt[e] - zmax);
            for (j = 0; j < k; ++j) wts[(size_t)t * k + j] = exp(zt[ids[(size_t)t * k + j]] - zmax) / sum;
        }
    }
    free(taken);
}

/* ------------------------------------------------------------------------ */
/* Expert FFN (SwiGLU) and the unpaged layer                                 */
/* ------------------------------------------------------------------------ */

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* An expert is a gate, an up and a down projection [EXPLAINER, "The bus
 * problem"]: gate and up map hidden -> intermediate, down maps back;
 * a = silu(gate x) * (up x), y = down a. */
int orc_expert_ffn(int fmt, const uint8_t* record, int H, int I, const double* x, double* y) {
    size_t gu_bytes = orc_matrix_bytes(fmt, I, H);
    size_t dn_bytes = orc_matrix_bytes(fmt, H, I);
    const uint8_t* gate = record;
    const uint8_t* up = record + gu_bytes;
    const uint8_t* down = record + 2 * gu_bytes;
    double g_gate = 1.0, g_up = 1.0, g_down = 1.0;
    double *w, *a;
    int i, h, c;
    if (gu_bytes == 0 || dn_bytes == 0) return ORC_ERR_INVALID;
    if (fmt == ORC_FMT_NVFP4) {
        const uint8_t* gl = down + dn_bytes;
        g_gate = rdf32(gl);
        g_up = rdf32(gl + 4);
        g_down = rdf32(gl + 8);
    }
    w = (double*)malloc(sizeof(double) * (size_t)(H > I ? H : I));
    a = (double*)malloc(sizeof(double) * (size_t)I);
    for (i = 0; i < I; ++i) {
        double gsum = 0.0, usum = 0.0;
        dequant_row(fmt, gate, I, H, g_gate, i, w);
        for (c = 0; c < H; ++c) gsum = gsum + w[c] * x[c];
        dequant_row(fmt, up, I, H, g_up, i, w);
        for (c = 0; c < H; ++c) usum = usum + w[c] * x[c];
        a[i] = silu(gsum) * usum;
    }
    for (h = 0; h < H; ++h) {
        double acc = 0.0;
        dequant_row(fmt, down, H, I, g_down, h, w);
        for (c = 0; c < I; ++c) acc = acc + w[c] * a[c];
        y[h] = acc;
    }
    free(w);
    free(a);
    return ORC_OK;
}

/* The layer with no cache at all: every expert read straight from its host
 * record. Paging leaves routing alone, so the paged layer must give this
 * same result [PAGED, "Can paging change the model's outputs?"]. Output =
 * sum over the k picks of weight * expert(x), in rank order, plus the
 * always-on shared expert with weight 1 (ten routed experts plus one shared
 * per token in [EXPLAINER, "The model that should not fit"]). */
int orc_moe_layer(int fmt, int H, int I, int E, int k, int norm,
                  const uint8_t* const* records, const uint8_t* shared_record,
                  const uint16_t* x_bf16, int T, const uint16_t* router_w_bf16,
                  const float* router_bias, int32_t* ids, double* wts, double* y) {
    double* z = (double*)malloc(sizeof(double) * (size_t)T * E);
    double* x = (double*)malloc(sizeof(double) * (size_t)H);
    double* ye = (double*)malloc(sizeof(double) * (size_t)H);
    int t, j, h, rc = ORC_OK;
    orc_router_logits(x_bf16, T, H, router_w_bf16, E, router_bias, z);
    orc_topk(z, T, E, k, norm, ids, wts);
    for (t = 0; t < T && rc == ORC_OK; ++t) {
        double* yt = y + (size_t)t * H;
        for (h = 0; h < H; ++h) x[h] = orc_decode_bf16(x_bf16[(size_t)t * H + h]);
        for (h = 0; h < H; ++h) yt[h] = 0.0;
        for (j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            double wt = wts[(size_t)t * k + j];
            if (!records || !records[e]) { rc = ORC_ERR_MISSING; break; }
            rc = orc_expert_ffn(fmt, records[e], H, I, x, ye);
            if (rc != ORC_OK) break;
            for (h = 0; h < H; ++h) yt[h] = yt[h] + wt * ye[h];
        }
        if (rc == ORC_OK && shared_record) {
            rc = orc_expert_ffn(fmt, shared_record, H, I, x, ye);
            for (h = 0; h < H; ++h) yt[h] = yt[h] + ye[h];
        }
    }
    free(z);
    free(x);
    free(ye);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* The literal LRU list                                                      */
/* ------------------------------------------------------------------------ */

/* State per [EXPLAINER, "Inside llama.cpp PR #29887"]: a slot map per layer
 * (expert -> slot, -1 when absent), the reverse map key_of (slot -> layer*E +
 * expert, -1 when empty), and a doubly linked list over the slots of a pool
 * whose head is the least recently used slot and whose tail the most
 * recently used. With one pool per layer the pool is that layer's K-slot
 * table [PAGED, "What does Paged Experts actually do?"]; with a shared pool
 * the layers compete for slots, so an expert of one layer may evict an
 * expert of another [T4, "What the MoE Cache Actually Caches"]. */
struct orc_cache {
    int L, E, mode, K, n_pools, max_cache_tokens;
    double slot_bytes;
    int32_t* slot_map; /* [L*E] */
    int32_t* key_of;   /* [n_pools*K] */
    int32_t* prev;     /* [n_pools*K] */
    int32_t* next;     /* [n_pools*K] */
    int32_t* head;     /* [n_pools] */
    int32_t* tail;     /* [n_pools] */
    uint64_t stats[3][4];
    char* seen;      /* [E] scratch */
    int32_t* uniq;   /* [E] scratch */
    char* was_hit;   /* [E] scratch */
    int policy;      /* ORC_POLICY_LRU or ORC_POLICY_LFU */
    uint64_t* uses;  /* [L*E] calls that routed each key, over the whole history (LFU) */
    char* inuse;     /* [K] scratch: slots the current call holds (LFU) */
    int prefill_mode;   /* ORC_PREFILL_READ_ONLY or ORC_PREFILL_PAGE_IN */
    int32_t* use_slot;  /* [E] scratch: the slot an expert is read from in the current call */
    /* adaptive per-layer capacity (per-layer pools): each pool's array has K
     * places, of which Kp[p] are its slots (active[p*K + s]); K0 slots each at
     * the start; every period*L decode calls capacity moves (see
     * orc_cache_set_adaptive) */
    int K0;
    int32_t* Kp;          /* [n_pools] */
    char* active;         /* [n_pools*K] */
    int adapt_period, adapt_step, adapt_kmin;
    uint64_t decode_calls;
    uint64_t* win;        /* [L][2] hits, misses of decode calls since the last move */
};

/* Initial list: every slot empty, ordered 0..K0-1 with slot 0 at the head
 * (places K0..K-1 of an adaptive pool hold no slot yet). */
void orc_cache_reset(orc_cache* c) {
    int p, s;
    for (s = 0; s < c->L * c->E; ++s) c->slot_map[s] = -1;
    for (p = 0; p < c->n_pools; ++p) {
        int32_t* pv = c->prev + (size_t)p * c->K;
        int32_t* nx = c->next + (size_t)p * c->K;
        for (s = 0; s < c->K; ++s) {
            c->key_of[(size_t)p * c->K + s] = -1;
            c->active[(size_t)p * c->K + s] = s < c->K0;
            pv[s] = s < c->K0 ? s - 1 : -1;
            nx[s] = (s + 1 < c->K0) ? s + 1 : -1;
        }
        c->head[p] = 0;
        c->tail[p] = c->K0 - 1;
        c->Kp[p] = c->K0;
    }
    memset(c->stats, 0, sizeof(c->stats));
    memset(c->uses, 0, sizeof(uint64_t) * (size_t)c->L * c->E);
    memset(c->win, 0, sizeof(uint64_t) * 2 * (size_t)c->L);
    c->decode_calls = 0;
}

orc_cache* orc_cache_create(int L, int E, int pool_mode, int slots_per_pool, double slot_bytes,
                            int max_cache_tokens) {
    orc_cache* c;
    if (L <= 0 || E <= 0 || slots_per_pool <= 0) return NULL;
    if (pool_mode != ORC_POOL_PER_LAYER && pool_mode != ORC_POOL_SHARED) return NULL;
    c = (orc_cache*)calloc(1, sizeof(orc_cache));
    c->L = L;
    c->E = E;
    c->mode = pool_mode;
    c->K = slots_per_pool;
    c->n_pools = pool_mode == ORC_POOL_SHARED ? 1 : L;
    c->max_cache_tokens = max_cache_tokens;
    c->slot_bytes = slot_bytes;
    c->slot_map = (int32_t*)malloc(sizeof(int32_t) * (size_t)L * E);
    c->key_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->n_pools * c->K);
    c->prev = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->n_pools * c->K);
    c->next = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->n_pools * c->K);
    c->head = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->n_pools);
    c->tail = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->n_pools);
    c->seen = (char*)malloc((size_t)E);
    c->uniq = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    c->was_hit = (char*)malloc((size_t)E);
    c->uses = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)L * E);
    c->inuse = (char*)malloc((size_t)c->K);
    c->use_slot = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    c->K0 = c->K;
    c->Kp = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->n_pools);
    c->active = (char*)malloc((size_t)c->n_pools * c->K);
    c->win = (uint64_t*)malloc(sizeof(uint64_t) * 2 * (size_t)L);
    c->policy = ORC_POLICY_LRU;
    c->prefill_mode = ORC_PREFILL_READ_ONLY;
    orc_cache_reset(c);
    return c;
}

/* Eviction policy. LRU is the page's [EXPLAINER, "Inside llama.cpp PR
 * #29887"]. LFU is the frequency policy of [EXPLAINER, "How MoE expert
 * offloading works with an LRU expert cache"] (its toy table's LFU column)
 * and [FP4LOCAL, "Decode"] ("least frequently used eviction"); neither page
 * prints its rule. Reading taken: every key counts the calls that routed it
 * over the whole history (evicted or not); a miss takes, among the slots the
 * call does not hold, the one whose key has the fewest uses (an empty slot
 * first), the least recently used on ties. Counting over the whole history
 * is what makes the toy's LFU hit rate the probability mass of its most
 * popular experts, as its column shows. Changing the policy resets the
 * cache. */
int orc_cache_set_policy(orc_cache* c, int policy) {
    if (!c || (policy != ORC_POLICY_LRU && policy != ORC_POLICY_LFU)) return ORC_ERR_INVALID;
    if (policy != ORC_POLICY_LRU && c->prefill_mode == ORC_PREFILL_PAGE_IN) return ORC_ERR_INVALID;
    c->policy = policy;
    orc_cache_reset(c);
    return ORC_OK;
}

/* How a prefill call (T > max_cache_tokens) treats the cache. The pages
 * differ [T4, "What the MoE Cache Actually Caches"; PAGED, "Why do short
 * prompts get slower first tokens?"]:
 *  - READ_ONLY (llama.cpp): resident experts are read in place, the others
 *    are staged for the call only; the list does not change.
 *  - PAGE_IN (SGLang Paged Experts): the prefill pages in every expert it
 *    routes to that is not resident, once. Read as the decode transaction
 *    over all of the call's distinct experts, without the capacity rule:
 *    dedupe, touch the hits, then each miss in ascending order takes the
 *    least recently used slot, evicting its key, and becomes the most
 *    recently used. When the call has more distinct experts than slots, the
 *    later misses take slots that earlier experts of the same call were read
 *    from (so each such expert is used, and then evicted, within the call).
 *    Needs LRU eviction (the LFU rule takes slots the call does not hold).
 * ORC_ERR_INVALID for another value, or PAGE_IN with LFU. */
int orc_cache_set_prefill_mode(orc_cache* c, int mode) {
    if (!c || (mode != ORC_PREFILL_READ_ONLY && mode != ORC_PREFILL_PAGE_IN)) return ORC_ERR_INVALID;
    if (mode == ORC_PREFILL_PAGE_IN && c->policy != ORC_POLICY_LRU) return ORC_ERR_INVALID;
    c->prefill_mode = mode;
    return ORC_OK;
}

/* Adaptive per-layer capacity [FP4LOCAL, "Decode"]: "some capacity is moved
 * from layers with high hit rates to layers with low hit rates" as decoding
 * progresses, with the same total. The page prints no rule; reading taken:
 * per-layer pools; every period * L decode calls (each wave a call; prefill
 * calls do not count), the layer whose decode calls since the last move had
 * the highest hit rate (hits / (hits + misses)) gives `step` slots, one at a
 * time, to the layer with the lowest, lower layer first on ties (rates are
 * compared exactly, h1 (h2 + m2) against h2 (h1 + m1)), layers without a
 * decode call in the window taking no part; the giver keeps at least kmin
 * slots and the taker at most kmax. A moved slot is the giver's least
 * recently used one, its expert evicted; it becomes the taker's empty least
 * recently used slot, at the lowest place of its array that holds no slot.
 * No move when the two rates are equal. The window then restarts. */
int orc_cache_set_adaptive(orc_cache* c, int period, int step, int kmin, int kmax) {
    int32_t *ko, *pv, *nx;
    char *in, *ac;
    if (!c || c->mode != ORC_POOL_PER_LAYER || period < 1 || step < 1 || kmin < 1 || kmin > c->K0 ||
        kmax < c->K0)
        return ORC_ERR_INVALID;
    ko = (int32_t*)realloc(c->key_of, sizeof(int32_t) * (size_t)c->n_pools * kmax);
    pv = (int32_t*)realloc(c->prev, sizeof(int32_t) * (size_t)c->n_pools * kmax);
    nx = (int32_t*)realloc(c->next, sizeof(int32_t) * (size_t)c->n_pools * kmax);
    in = (char*)realloc(c->inuse, (size_t)kmax);
    ac = (char*)realloc(c->active, (size_t)c->n_pools * kmax);
    if (!ko || !pv || !nx || !in || !ac) return ORC_ERR_INVALID;
    c->key_of = ko;
    c->prev = pv;
    c->next = nx;
    c->inuse = in;
    c->active = ac;
    c->K = kmax;
    c->adapt_period = period;
    c->adapt_step = step;
    c->adapt_kmin = kmin;
    orc_cache_reset(c);
    return ORC_OK;
}

/* One slot from pool d to pool r (adaptive capacity). */
static void adapt_move(orc_cache* c, int d, int r) {
    int32_t* pv = c->prev + (size_t)d * c->K;
    int32_t* nx = c->next + (size_t)d * c->K;
    const int32_t s = c->head[d];
    const int32_t key = c->key_of[(size_t)d * c->K + s];
    int32_t t;
    if (key >= 0) c->slot_map[key] = -1;
    c->key_of[(size_t)d * c->K + s] = -1;
    c->head[d] = nx[s];
    if (nx[s] >= 0) pv[nx[s]] = -1;
    else c->tail[d] = -1;
    c->active[(size_t)d * c->K + s] = 0;
    c->Kp[d]--;
    for (t = 0; c->active[(size_t)r * c->K + t]; ++t) {
    }
    pv = c->prev + (size_t)r * c->K;
    nx = c->next + (size_t)r * c->K;
    c->active[(size_t)r * c->K + t] = 1;
    c->key_of[(size_t)r * c->K + t] = -1;
    pv[t] = -1;
    nx[t] = c->head[r];
    if (c->head[r] >= 0) pv[c->head[r]] = t;
    else c->tail[r] = t;
    c->head[r] = t;
    c->Kp[r]++;
}

static void adapt_after_call(orc_cache* c) {
    int l, d = -1, r = -1, i;
    if (!c->adapt_period) return;
    c->decode_calls++;
    if (c->decode_calls % ((uint64_t)c->adapt_period * c->L) != 0) return;
    for (l = 0; l < c->L; ++l) {
        const uint64_t h = c->win[2 * l], m = c->win[2 * l + 1];
        if (h + m == 0) continue;
        if (c->Kp[l] - c->adapt_step >= c->adapt_kmin &&
            (d < 0 || h * (c->win[2 * d] + c->win[2 * d + 1]) > c->win[2 * d] * (h + m)))
            d = l;
        if (c->Kp[l] + c->adapt_step <= c->K &&
            (r < 0 || h * (c->win[2 * r] + c->win[2 * r + 1]) < c->win[2 * r] * (h + m)))
            r = l;
    }
    if (d >= 0 && r >= 0 && d != r &&
        c->win[2 * d] * (c->win[2 * r] + c->win[2 * r + 1]) > c->win[2 * r] * (c->win[2 * d] + c->win[2 * d + 1]))
        for (i = 0; i < c->adapt_step; ++i) adapt_move(c, d, r);
    memset(c->win, 0, sizeof(uint64_t) * 2 * (size_t)c->L);
}

int orc_cache_pool_slots(const orc_cache* c, int pool) {
    return (!c || pool < 0 || pool >= c->n_pools) ? -1 : c->Kp[pool];
}

void orc_cache_destroy(orc_cache* c) {
    if (!c) return;
    free(c->use_slot);
    free(c->Kp);
    free(c->active);
    free(c->win);
    free(c->slot_map);
    free(c->key_of);
    free(c->prev);
    free(c->next);
    free(c->head);
    free(c->tail);
    free(c->seen);
    free(c->uniq);
    free(c->was_hit);
    free(c->uses);
    free(c->inuse);
    free(c);
}

/* Move slot s of pool p to the most-recently-used end in O(1): unlink it
 * from its neighbours, then append it after the current tail. */
static void lru_touch(orc_cache* c, int p, int32_t s) {
    int32_t* pv = c->prev + (size_t)p * c->K;
    int32_t* nx = c->next + (size_t)p * c->K;
    int32_t before, after;
    if (s == c->tail[p]) return; /* already most recent */
    before = pv[s];
    after = nx[s]; /* exists, since s is not the tail */
    if (before >= 0) nx[before] = after;
    else c->head[p] = after;
    pv[after] = before;
    pv[s] = c->tail[p];
    nx[s] = -1;
    nx[c->tail[p]] = s;
    c->tail[p] = s;
}

static int cmp_i32(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

static int bucket_of(int T) { return T <= 8 ? 0 : (T <= 32 ? 1 : 2); }

/* One layer call [EXPLAINER, "Inside llama.cpp PR #29887"]:
 *  1. the routed ids are deduplicated, keeping the first occurrence in
 *     [token][rank] order (the page elides this step; this order is our
 *     reading);
 *  2. every resident expert is touched, in that order, so the head can only
 *     hold a slot this call does not use;
 *  3. the misses are sorted ascending; each takes the head slot, evicts the
 *     key that slot held (its slot map entry becomes -1), records the new
 *     key, is touched, and is appended to the fill list.
 * More distinct experts than slots is refused before anything changes (the
 * page aborts there; we return an error). Batches above the cache limit do
 * not go through the cache transaction [T4, "What the MoE Cache Actually
 * Caches"; EXPLAINER, "The rules in the code"]: they only look up what is
 * resident. */
int orc_cache_plan(orc_cache* c, int layer, const int32_t* ids, int n_ids, int T,
                   int32_t* slot_of, uint8_t* hit_of, int32_t* fill_expert, int32_t* fill_slot,
                   int* n_fill, int* n_hit, int* n_uniq) {
    int i, nu = 0, nh = 0, nf = 0, p, b;
    int32_t* smap;
    if (!c || layer < 0 || layer >= c->L || n_ids < 0 || T <= 0) return ORC_ERR_INVALID;
    for (i = 0; i < n_ids; ++i)
        if (ids[i] < 0 || ids[i] >= c->E) return ORC_ERR_INVALID;
    smap = c->slot_map + (size_t)layer * c->E;
    p = c->mode == ORC_POOL_SHARED ? 0 : layer;

    memset(c->seen, 0, (size_t)c->E);
    memset(c->was_hit, 0, (size_t)c->E);
    for (i = 0; i < n_ids; ++i) {
        if (!c->seen[ids[i]]) {
            c->seen[ids[i]] = 1;
            c->uniq[nu++] = ids[i];
        }
    }
    b = bucket_of(T);

    if (T > c->max_cache_tokens && c->prefill_mode == ORC_PREFILL_PAGE_IN) {
        /* page-in: the decode transaction over every distinct expert, with
         * no capacity rule; slot_of is the slot each expert is read from
         * (a hit's slot when it is touched, a miss's when it is filled) */
        for (i = 0; i < nu; ++i) {
            int32_t e = c->uniq[i];
            if (smap[e] >= 0) {
                c->use_slot[e] = smap[e];
                lru_touch(c, p, smap[e]);
                c->was_hit[e] = 1;
                nh++;
            }
        }
        qsort(c->uniq, (size_t)nu, sizeof(int32_t), cmp_i32);
        for (i = 0; i < nu; ++i) {
            int32_t e = c->uniq[i], s, old;
            if (c->was_hit[e]) continue;
            s = c->head[p];
            old = c->key_of[(size_t)p * c->K + s];
            if (old >= 0) c->slot_map[old] = -1;
            c->key_of[(size_t)p * c->K + s] = layer * c->E + e;
            smap[e] = s;
            lru_touch(c, p, s);
            c->use_slot[e] = s;
            fill_expert[nf] = e;
            fill_slot[nf] = s;
            nf++;
        }
        for (i = 0; i < n_ids; ++i) {
            slot_of[i] = c->use_slot[ids[i]];
            hit_of[i] = (uint8_t)c->was_hit[ids[i]];
        }
        c->stats[b][0] += 1;
        c->stats[b][1] += (uint64_t)nh;
        c->stats[b][2] += (uint64_t)nf;
        c->stats[b][3] += (uint64_t)((double)nf * c->slot_bytes);
        *n_fill = nf;
        *n_hit = nh;
        *n_uniq = nu;
        return ORC_OK;
    }

    if (T > c->max_cache_tokens) {
        /* read-only lookup: resident experts are read in place, the rest are
         * staged for this call only */
        for (i = 0; i < nu; ++i)
            if (smap[c->uniq[i]] >= 0) { c->was_hit[c->uniq[i]] = 1; nh++; }
        for (i = 0; i < n_ids; ++i) {
            slot_of[i] = smap[ids[i]];
            hit_of[i] = (uint8_t)c->was_hit[ids[i]];
        }
        c->stats[b][0] += 1;
        c->stats[b][1] += (uint64_t)nh;
        c->stats[b][2] += (uint64_t)(nu - nh);
        c->stats[b][3] += (uint64_t)((double)(nu - nh) * c->slot_bytes);
        *n_fill = 0;
        *n_hit = nh;
        *n_uniq = nu;
        return ORC_OK;
    }

    if (nu > c->Kp[p]) return ORC_ERR_CAPACITY;

    if (c->policy == ORC_POLICY_LFU) {
        memset(c->inuse, 0, (size_t)c->K);
        for (i = 0; i < nu; ++i) c->uses[(size_t)layer * c->E + c->uniq[i]] += 1;
    }
    for (i = 0; i < nu; ++i) {
        int32_t e = c->uniq[i];
        if (smap[e] >= 0) {
            lru_touch(c, p, smap[e]);
            if (c->policy == ORC_POLICY_LFU) c->inuse[smap[e]] = 1;
            c->was_hit[e] = 1;
            nh++;
        }
    }
    qsort(c->uniq, (size_t)nu, sizeof(int32_t), cmp_i32);
    for (i = 0; i < nu; ++i) {
        int32_t e = c->uniq[i];
        int32_t s, old;
        if (c->was_hit[e]) continue;
        s = c->head[p];
        if (c->policy == ORC_POLICY_LFU) {
            /* walk the list from its least recent end; keep the first slot
             * with the fewest uses among those the call does not hold */
            int32_t q = c->head[p], best = -1;
            double best_uses = 0.0;
            while (q >= 0) {
                if (!c->inuse[q]) {
                    const int32_t key = c->key_of[(size_t)p * c->K + q];
                    const double u = key < 0 ? -1.0 : (double)c->uses[key];
                    if (best < 0 || u < best_uses) { best = q; best_uses = u; }
                }
                q = c->next[(size_t)p * c->K + q];
            }
            s = best;
            c->inuse[s] = 1;
        }
        old = c->key_of[(size_t)p * c->K + s];
        if (old >= 0) c->slot_map[old] = -1; /* key = layer*E + expert */
        c->key_of[(size_t)p * c->K + s] = layer * c->E + e;
        smap[e] = s;
        lru_touch(c, p, s);
        fill_expert[nf] = e;
        fill_slot[nf] = s;
        nf++;
    }
    for (i = 0; i < n_ids; ++i) {
        slot_of[i] = smap[ids[i]];
        hit_of[i] = (uint8_t)c->was_hit[ids[i]];
    }
    /* counters per [EXPLAINER, "Inside llama.cpp PR #29887"] (hits, misses,
     * bytes uploaded), bucketed by batch size as the log line is [T4,
     * "Without Reading Logs"]: <= 8 tokens, 9-32, larger. */
    c->stats[b][0] += 1;
    c->stats[b][1] += (uint64_t)nh;
    c->stats[b][2] += (uint64_t)nf;
    c->stats[b][3] += (uint64_t)((double)nf * c->slot_bytes);
    *n_fill = nf;
    *n_hit = nh;
    *n_uniq = nu;
    c->win[2 * layer] += (uint64_t)nh;
    c->win[2 * layer + 1] += (uint64_t)nf;
    adapt_after_call(c);
    return ORC_OK;
}

void orc_cache_state(const orc_cache* c, int32_t* slot_map, int32_t* key_of, int32_t* order) {
    int p, s, n;
    if (slot_map) memcpy(slot_map, c->slot_map, sizeof(int32_t) * (size_t)c->L * c->E);
    if (key_of) memcpy(key_of, c->key_of, sizeof(int32_t) * (size_t)c->n_pools * c->K);
    if (order) {
        for (p = 0; p < c->n_pools; ++p) {
            const int32_t* nx = c->next + (size_t)p * c->K;
            n = 0;
            for (s = c->head[p]; s >= 0 && n < c->K; s = nx[s]) order[(size_t)p * c->K + n++] = s;
            for (; n < c->K; ++n) order[(size_t)p * c->K + n] = -1; /* broken list */
        }
    }
}

int orc_cache_num_pools(const orc_cache* c) { return c->n_pools; }
int orc_cache_slots(const orc_cache* c) { return c->K; }

void orc_cache_stats(const orc_cache* c, uint64_t* stats) {
    int b, j;
    for (b = 0; b < 3; ++b)
        for (j = 0; j < 4; ++j) stats[b * 4 + j] = c->stats[b][j];
}

/* Waves of a decode step [PAGED, "What happens with more than one request?"]:
 * a step is served by one wave only if tokens x top_k <= K, that is up to
 * K // top_k tokens; a larger step needs several waves, each with its own
 * page-in. The page does not say how the tokens are grouped; the plainest
 * reading, taken here, is successive groups of K // top_k tokens in token
 * order, the last one shorter. Writes each wave's first token and token
 * count; returns the number of waves, or 0 when K < top_k (no wave fits). */
int orc_wave_split(int T, int k, int K, int32_t* start, int32_t* count) {
    int per, n = 0, t0;
    if (T < 1 || k < 1 || K < k) return 0;
    per = K / k;
    for (t0 = 0; t0 < T; t0 += per) {
        start[n] = t0;
        count[n] = (T - t0 < per) ? T - t0 : per;
        n++;
    }
    return n;
}

/* Consecutive experts going to consecutive slots move as one copy
 * [EXPLAINER, "Inside llama.cpp PR #29887"]. */
int orc_count_runs(const int32_t* fill_expert, const int32_t* fill_slot, int n_fill) {
    int i = 0, runs = 0;
    while (i < n_fill) {
        int n = 1;
        while (i + n < n_fill && fill_expert[i + n] == fill_expert[i] + n && fill_slot[i + n] == fill_slot[i] + n) n++;
        runs++;
        i += n;
    }
    return runs;
}
