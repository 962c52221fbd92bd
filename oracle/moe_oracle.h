/*
 * moe_oracle.h -- CPU oracle for a routed mixture-of-experts FFN layer that
 * runs over an LRU expert cache.
 *
 * TEST INFRASTRUCTURE. This library is the slow, plain, obviously-correct
 * statement of what the GPU path must compute. Only the test suite, the
 * package smoke check and the benchmark's CPU-baseline leg may load it. The
 * product (the CUDA library under paged_expert_cache_gb300/) never includes,
 * links or calls anything here, and nothing here includes product headers.
 *
 * All floating point is fp64, single threaded, built with -ffp-contract=off
 * so that no multiply-add is fused behind the reader's back.
 *
 * Pages followed (cited by title and section):
 *  [EXPLAINER] "Your GPU holds 24 GB. This model is 94 GB. It still runs."
 *              (cloudmash.blog), sections "The bus problem", "How MoE expert
 *              offloading works with an LRU expert cache", "Inside llama.cpp
 *              PR #29887: slot maps, banks, and only the misses cross PCIe",
 *              "The rules in the code".
 *  [PAGED]     "Running an MoE Model Larger Than Your VRAM: SGLang Paged
 *              Experts, the PCIe Math, and the 4-Request Cliff" (dev.to),
 *              sections "What does Paged Experts actually do?", "Can paging
 *              change the model's outputs?", "A preflight script".
 *  [T4]        "llama.cpp MoE Cache Benchmark: Doubling 30B Model Decode Speed
 *              on a T4" (kongchang.com), sections "What the MoE Cache Actually
 *              Caches", "Without Reading Logs, You Won't Know the Hit Rate".
 *  [FP4LOCAL]  "Running a 95 GiB MoE Model on a 32 GiB GPU" (busyjay.com),
 *              sections "Decode", "Prefill".
 *  [NVME]      "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by
 *              streaming experts from NVMe" (atlasrepo.com), section
 *              "Workflow".
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight formats of an expert record (numeric values are the interface's). */
enum { ORC_FMT_BF16 = 0, ORC_FMT_Q4_0 = 1, ORC_FMT_FP8_B128 = 2, ORC_FMT_NVFP4 = 3 };
/* Pool scopes: one K-slot pool per layer [PAGED], or one pool for all layers [T4]. */
enum { ORC_POOL_PER_LAYER = 0, ORC_POOL_SHARED = 1 };
enum { ORC_POLICY_LRU = 0, ORC_POLICY_LFU = 1 };
enum { ORC_PREFILL_READ_ONLY = 0, ORC_PREFILL_PAGE_IN = 1 };
/* Status codes. */
enum { ORC_OK = 0, ORC_ERR_INVALID = 1, ORC_ERR_CAPACITY = 2, ORC_ERR_MISSING = 3 };

/* ---- scalar decoders, each written from its format definition ---- */
double orc_decode_fp16(uint16_t bits);  /* IEEE-754 binary16 */
double orc_decode_bf16(uint16_t bits);  /* upper half of IEEE-754 binary32 */
double orc_decode_e4m3(uint8_t bits);   /* OCP FP8 E4M3 (no infinities, S.1111.111 = NaN) */
double orc_decode_e2m1(uint8_t nibble); /* OCP FP4 E2M1 (low 4 bits used) */
/* kind: 0 fp16, 1 bf16 (16-bit inputs); 2 e4m3, 3 e2m1 (8-bit inputs). */
int orc_decode_array(int kind, const void* in, size_t n, double* out);

/* ---- record geometry ---- */
/* Canonical bytes of one matrix of `rows` outputs by `cols` inputs. */
size_t orc_matrix_bytes(int fmt, int rows, int cols);
/* Canonical expert record: gate [I x H], up [I x H], down [H x I]; NVFP4 adds
 * three fp32 global scales (gate, up, down) at the end. */
size_t orc_record_bytes(int fmt, int H, int I);
/* Bytes a cache slot holds (the record without the NVFP4 global scales). */
size_t orc_slot_bytes(int fmt, int H, int I);
/* Slots a pool of pool_bytes buys: floor(pool_bytes / slot_bytes). */
int64_t orc_slots_for_budget(double pool_bytes, double slot_bytes);

/* Dequantise a whole canonical matrix into out[rows*cols] (row-major).
 * g is the NVFP4 global scale (ignored by the other formats). */
int orc_dequant_matrix(int fmt, const uint8_t* mat, int rows, int cols, double g, double* out);

/* ---- router ---- */
/* z[t*E+e] = sum_h x[t,h]*W[e,h] (ascending h, fp64, unfused) + bias[e]. */
void orc_router_logits(const uint16_t* x_bf16, int T, int H, const uint16_t* w_bf16, int E,
                       const float* bias /* may be NULL */, double* z);
/* Top-k by logit, ties to the lower expert id; ids in rank order.
 * norm != 0: weights are the softmax over the k selected logits;
 * norm == 0: weights are the full softmax over all E, read at the selected. */
void orc_topk(const double* z, int T, int E, int k, int norm, int32_t* ids, double* wts);

/* ---- expert FFN and the plain (unpaged) layer ---- */
/* y[H] = down * (silu(gate*x) .* (up*x)) for one canonical record. */
int orc_expert_ffn(int fmt, const uint8_t* record, int H, int I, const double* x, double* y);
/* The whole layer with every expert read straight from its host record:
 * routing, weights, weighted sum over the k picks in rank order, plus the
 * shared expert (weight 1) when shared_record != NULL. records[e] may be NULL
 * for experts no token selects (ORC_ERR_MISSING otherwise). */
int orc_moe_layer(int fmt, int H, int I, int E, int k, int norm,
                  const uint8_t* const* records, const uint8_t* shared_record,
                  const uint16_t* x_bf16, int T, const uint16_t* router_w_bf16,
                  const float* router_bias, int32_t* ids, double* wts, double* y);

/* ---- the literal LRU list ---- */
typedef struct orc_cache orc_cache;
orc_cache* orc_cache_create(int L, int E, int pool_mode, int slots_per_pool, double slot_bytes,
                            int max_cache_tokens);
void orc_cache_destroy(orc_cache* c);
void orc_cache_reset(orc_cache* c);
/* One layer call of T tokens with ids[n_ids] in [token][rank] order.
 * T <= max_cache_tokens: the cache transaction (dedupe, touch hits, sorted
 *   misses take the LRU head). T > max_cache_tokens: read-only lookup (no
 *   list change); misses are staged, not cached, and slot_of is -1 for them;
 *   or, in ORC_PREFILL_PAGE_IN mode, the transaction over every distinct
 *   expert without the capacity rule (slot_of: the slot each is read from).
 * Outputs: slot_of[n_ids], hit_of[n_ids] (1 if that id's expert was resident
 * at the start of the call), fill_expert/fill_slot[n_fill], counts. Returns
 * ORC_ERR_CAPACITY (state untouched) if the unique count exceeds the pool. */
int orc_cache_plan(orc_cache* c, int layer, const int32_t* ids, int n_ids, int T,
                   int32_t* slot_of, uint8_t* hit_of, int32_t* fill_expert, int32_t* fill_slot,
                   int* n_fill, int* n_hit, int* n_uniq);
/* Copies of the state: slot_map[L*E], key_of[n_pools*K], and the list order
 * of each pool from least to most recently used: order[n_pools*K]. */
void orc_cache_state(const orc_cache* c, int32_t* slot_map, int32_t* key_of, int32_t* order);
int orc_cache_num_pools(const orc_cache* c);
int orc_cache_slots(const orc_cache* c);
/* stats[bucket*4 + {0 calls, 1 hits, 2 misses, 3 bytes}], buckets: T<=8, 9..32, >32. */
void orc_cache_stats(const orc_cache* c, uint64_t* stats);
/* Eviction policy (ORC_POLICY_LRU, the default, or ORC_POLICY_LFU); resets the
 * cache. ORC_ERR_INVALID for another value. */
int orc_cache_set_policy(orc_cache* c, int policy);
/* Prefill mode (ORC_PREFILL_READ_ONLY, the default, or ORC_PREFILL_PAGE_IN,
 * which needs LRU). ORC_ERR_INVALID otherwise. */
int orc_cache_set_prefill_mode(orc_cache* c, int mode);
/* Adaptive per-layer capacity (per-layer pools): every period * L decode
 * calls, `step` slots move, one at a time, from the layer with the highest
 * hit rate since the last move to the one with the lowest, within
 * [kmin, kmax] slots per layer; a moved slot leaves as its giver's least
 * recently used (expert evicted) and arrives as the taker's empty least
 * recently used, at the lowest free place of its array of kmax places.
 * Resets the cache. ORC_ERR_INVALID for a shared pool or bad bounds. */
int orc_cache_set_adaptive(orc_cache* c, int period, int step, int kmin, int kmax);
/* Slots pool `pool` holds now. */
int orc_cache_pool_slots(const orc_cache* c, int pool);
/* The waves of a decode step of T tokens on a pool of K slots: successive
 * groups of K // k tokens; returns their number (0 if K < k). */
int orc_wave_split(int T, int k, int K, int32_t* start, int32_t* count);
/* Number of copies after merging runs where expert and slot both step by one. */
int orc_count_runs(const int32_t* fill_expert, const int32_t* fill_slot, int n_fill);

#ifdef __cplusplus
}
#endif
#endif
