/*
 * moe_cache.h -- C ABI of a routed mixture-of-experts FFN layer that runs over
 * a GPU-resident, deliberately capped LRU pool of expert slots (GB300, sm_103a).
 *
 * The operation follows these pages (cited by title and section):
 *  [EXPLAINER] "Your GPU holds 24 GB. This model is 94 GB. It still runs."
 *              (cloudmash.blog): "How MoE expert offloading works with an LRU
 *              expert cache", "Inside llama.cpp PR #29887: slot maps, banks,
 *              and only the misses cross PCIe", "The rules in the code".
 *  [PAGED]     "Running an MoE Model Larger Than Your VRAM: SGLang Paged
 *              Experts, the PCIe Math, and the 4-Request Cliff" (dev.to):
 *              "What does Paged Experts actually do?", "What happens with more
 *              than one request?", "Can paging change the model's outputs?".
 *  [T4]        "llama.cpp MoE Cache Benchmark: Doubling 30B Model Decode Speed
 *              on a T4" (kongchang.com): "What the MoE Cache Actually Caches",
 *              "Without Reading Logs, You Won't Know the Hit Rate".
 *  [FP4LOCAL]  "Running a 95 GiB MoE Model on a 32 GiB GPU" (busyjay.com):
 *              "Decode", "Prefill".
 *  [NVME]      "Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by
 *              streaming experts from NVMe" (atlasrepo.com): "Workflow".
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" must be CUDA device memory of the handle's
 *    device; pointers marked "host" are ordinary host memory.
 *  - bf16 values are passed as raw 16-bit patterns; the caller owns every
 *    buffer it passes and keeps ownership after the call returns.
 *  - The handle owns all memory it allocates (pinned host store, slot pool,
 *    tables, scratch) and frees it in moe_cache_destroy.
 *  - Calls on one handle must not overlap: issue them from one host thread
 *    and, for moe_layer_forward, on one stream (or order the streams).
 *  - Every entry point returns a moe_status_t; on failure a message is kept
 *    for moe_last_error. A CUDA error seen asynchronously is reported as
 *    MOE_ERR_CUDA by the next call that synchronises (stats, trace, state).
 */
#ifndef MOE_CACHE_H
#define MOE_CACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 3

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID = 1,   /* bad argument or configuration */
    MOE_ERR_CAPACITY = 2,  /* the call needs more slots than the pool has */
    MOE_ERR_CUDA = 3,      /* a CUDA runtime call or kernel failed */
    MOE_ERR_OOM = 4,       /* host or device allocation failed */
    MOE_ERR_STATE = 5,     /* the handle is not ready (e.g. experts not loaded) */
    MOE_ERR_TIMEOUT = 6    /* a bounded device-side wait gave up */
} moe_status_t;

/* Expert weight formats. Canonical host record = gate [I x H], up [I x H],
 * down [H x I] back to back (rows are output features, row-major):
 *  MOE_FMT_BF16     : bf16 weights, 2 bytes each.
 *  MOE_FMT_Q4_0     : per row, blocks of 32 consecutive weights, each block an
 *                     fp16 scale d (little-endian) then 16 bytes; byte i holds
 *                     weight i in its low nibble and weight i+16 in its high
 *                     nibble; w = d * (q - 8). 18 bytes per 32 weights, the
 *                     size [EXPLAINER, "The bus problem"] gives. cols % 32 == 0.
 *  MOE_FMT_FP8_B128 : e4m3 (OCP "FN") codes row-major, then fp32 scales over
 *                     128 x 128 tiles (row-major over the tile grid, partial
 *                     tiles at the edges); w = e4m3(q) * s[r/128][c/128].
 *  MOE_FMT_NVFP4    : e2m1 codes two per byte (low nibble = even column), then
 *                     one e4m3 scale per 16 consecutive weights of a row; the
 *                     record ends with three fp32 global scales (gate, up,
 *                     down); w = e2m1(q) * e4m3(s) * g. cols % 16 == 0.
 * The library repacks records into its own slot layout at load time; a slot
 * holds the record without the NVFP4 global scales (those stay resident). */
typedef enum { MOE_FMT_BF16 = 0, MOE_FMT_Q4_0 = 1, MOE_FMT_FP8_B128 = 2, MOE_FMT_NVFP4 = 3 } moe_format_t;

/* Pool scope: one K-slot pool per layer [PAGED, "What does Paged Experts
 * actually do?"], or one pool shared by all layers, so an expert of one layer
 * can evict an expert of another [T4, "What the MoE Cache Actually Caches"]. */
typedef enum { MOE_POOL_PER_LAYER = 0, MOE_POOL_SHARED = 1 } moe_pool_mode_t;

/* How misses reach their slots:
 *  MOE_UPLOAD_PULL   : a copy kernel on the forward's stream reads the mapped
 *                      pinned host store directly (no host round trip; the
 *                      whole forward can be captured in a CUDA graph).
 *  MOE_UPLOAD_MEMCPY : the host reads the fill list back (one stream sync per
 *                      call) and issues one cudaMemcpyAsync per merged run of
 *                      consecutive experts into consecutive slots [EXPLAINER,
 *                      "Inside llama.cpp PR #29887"]. */
typedef enum { MOE_UPLOAD_PULL = 0, MOE_UPLOAD_MEMCPY = 1 } moe_upload_mode_t;

/* How a decode call (T <= max_cache_tokens) is launched. The one-kernel path
 * runs the whole call as one persistent kernel (one CTA per SM, two bounded
 * grid-wide waits, the weight tiles streamed into shared memory by bulk
 * copies); it takes calls with T <= 8, T*k (+T shared) <= 48 and PULL
 * uploads whose shared-memory layout fits. The three-kernel path runs route,
 * gate/up and down kernels. */
typedef enum {
    MOE_DECODE_AUTO = 0,          /* one kernel for calls of one token, and of two tokens on
                                     per-layer pools (where it measured faster), three kernels
                                     otherwise */
    MOE_DECODE_THREE_KERNELS = 1, /* always three kernels */
    MOE_DECODE_ONE_KERNEL = 2     /* one kernel for every call that fits */
} moe_decode_mode_t;

/* Which slot a miss takes. LRU: the least recently used slot not held by the
 * call [EXPLAINER, "Inside llama.cpp PR #29887"]. LFU: a least frequently
 * used policy [FP4LOCAL, "Decode"]; the pages print no rule, so: every
 * (layer, expert) counts the decode calls that routed it over the whole
 * history, and a miss takes, among the slots its call does not hold, an empty
 * slot first, else the one whose expert has the fewest such calls, the least
 * recently used on ties. Counts saturate at 2^23. */
typedef enum {
    MOE_EVICT_LRU = 0,
    MOE_EVICT_LFU = 1
} moe_eviction_t;

/* What a prefill call (T > max_cache_tokens) does to the cache. The pages
 * differ:
 *  MOE_PREFILL_READ_ONLY : resident experts are read in place, the others
 *                          staged for the call only; the LRU order and the
 *                          slots do not change [T4, "What the MoE Cache
 *                          Actually Caches"].
 *  MOE_PREFILL_PAGE_IN   : the prefill pages in every expert it routes to
 *                          that is not resident, once [PAGED, "Why do short
 *                          prompts get slower first tokens?"]: the decode
 *                          transaction over all of the call's distinct
 *                          experts, without the capacity rule (hits touched
 *                          in first-occurrence order, then each miss in
 *                          ascending order takes the least recently used
 *                          slot; past K misses that is a slot the same call
 *                          read or filled, and only the last expert placed in
 *                          a slot stays). The records cross the host link
 *                          once, through the staging arena, and those that
 *                          stay are copied into their slots. Outputs are those
 *                          of MOE_PREFILL_READ_ONLY. Needs MOE_EVICT_LRU. */
typedef enum { MOE_PREFILL_READ_ONLY = 0, MOE_PREFILL_PAGE_IN = 1 } moe_prefill_mode_t;

typedef struct {
    int32_t num_layers;       /* L >= 1 */
    int32_t num_experts;      /* E routed experts per layer, 1..1024 */
    int32_t top_k;            /* k, 1..16 and <= E */
    int32_t hidden;           /* H, multiple of 64, at most 4096 */
    int32_t inter;            /* I, expert intermediate size, multiple of 64, at most 4096 */
    int32_t format;           /* moe_format_t */
    int32_t has_shared;       /* 1: an always-resident shared expert per layer */
    int32_t pool_mode;        /* moe_pool_mode_t */
    int32_t slots_per_layer;  /* K for MOE_POOL_PER_LAYER */
    int32_t upload_mode;      /* moe_upload_mode_t */
    double pool_bytes;        /* MOE_POOL_SHARED: slots = floor(pool_bytes / slot_bytes) */
    int32_t norm_topk;        /* 1: weights = softmax over the k picks; 0: full softmax */
    int32_t max_cache_tokens; /* calls with T above this skip the cache transaction (32) */
    int32_t prefill_group;    /* experts staged per prefill group (32) */
    int32_t max_tokens;       /* largest T of any call (sizes scratch) */
    int32_t device;           /* CUDA device ordinal */
    int32_t split_decode;     /* moe_decode_mode_t: how decode calls are launched (default
                                 MOE_DECODE_AUTO). Every mode gives bitwise identical results. */
    int32_t multi_wave;       /* 0 (default): a decode call with T * top_k above its pool's slots
                                 fails with MOE_ERR_CAPACITY. 1: it runs as successive waves of
                                 floor(slots / top_k) tokens (the last one shorter), each a cache
                                 transaction and a trace record of its own, in token order. */
    int32_t eviction;         /* moe_eviction_t (default MOE_EVICT_LRU) */
    int32_t speculate;        /* 0 (default) or 1: speculative next-layer routing and prefetch
                                 [NVME, "Workflow", "Evidence"]. A decode call of layer l with
                                 T <= 2 tokens, when layer l + 1's router is registered
                                 (moe_cache_set_router), ranks layer l + 1's experts on layer l's
                                 input on an internal side stream and copies the predicted ones that
                                 are not resident from the host store into a prefetch bank in device
                                 memory, beside layer l's expert kernels. Layer l + 1's call then
                                 reads its missed experts from the bank where they were predicted,
                                 instead of over the host link. Speculation moves bytes only: the
                                 routing, the cache plan, the outputs, the stats and the trace are
                                 bitwise those of speculate = 0. Decode calls take the three-kernel
                                 path while it is on. */
    int32_t prefill_mode;     /* moe_prefill_mode_t (default MOE_PREFILL_READ_ONLY) */
    int32_t adapt_period;     /* 0 (default): every layer keeps slots_per_layer slots. > 0 (per-layer
                                 pools): adaptive per-layer capacity [FP4LOCAL, "Decode": capacity
                                 moves from layers with high hit rates to layers with low hit
                                 rates, same total]. Every adapt_period * L decode calls (each wave
                                 a call; prefill calls do not count), adapt_step slots move, one at
                                 a time, from the layer whose decode calls since the last move had
                                 the highest hit rate to the one with the lowest (exact comparison,
                                 the lower layer first on ties; layers without a decode call in the
                                 window take no part; no move on equal rates), within
                                 [adapt_min_slots, adapt_max_slots] slots per layer. A moved slot
                                 leaves as the giver's least recently used (its expert evicted) and
                                 arrives as the taker's empty least recently used slot, at the
                                 lowest place of the taker's array that holds no slot. Each layer's
                                 array has adapt_max_slots places in device memory (the logical
                                 total stays L * slots_per_layer); the single-wave rule uses
                                 adapt_min_slots. */
    int32_t adapt_step;       /* slots per move (0: 1) */
    int32_t adapt_min_slots;  /* fewest slots a layer keeps (0: max(top_k, slots_per_layer / 2)) */
    int32_t adapt_max_slots;  /* most slots a layer holds (0: 2 * slots_per_layer - adapt_min_slots) */
} moe_config_t;

/* Fills cfg with defaults: norm_topk 1, max_cache_tokens 32, prefill_group 32,
 * max_tokens 32, upload PULL, per-layer pools, MOE_DECODE_AUTO, multi_wave 0,
 * MOE_EVICT_LRU, speculate 0, MOE_PREFILL_READ_ONLY, adapt_period 0; shape
 * fields zero. */
void moe_config_default(moe_config_t* cfg);

typedef struct {
    uint64_t calls;          /* layer calls in this bucket */
    uint64_t hits;           /* unique experts already resident, summed over calls */
    uint64_t misses;         /* unique experts uploaded (or staged, prefill) */
    uint64_t bytes_uploaded; /* misses * slot_bytes */
    uint64_t upload_ns;      /* device time spent in miss copies */
} moe_bucket_stats_t;

/* Buckets by tokens per call: [0] T <= 8, [1] 9..32, [2] > 32, as the
 * per-batch-size hit-rate log lines split them [T4, "Without Reading Logs"]. */
typedef struct {
    moe_bucket_stats_t bucket[3];
    int32_t num_pools;
    int32_t slots_per_pool;
    uint64_t slot_bytes;     /* bytes one slot holds */
    uint64_t record_bytes;   /* canonical record bytes */
    uint64_t topk_fp64_rerank; /* router calls that needed the fp64 re-rank */
    uint64_t spec_prefetched;  /* records copied into the prefetch bank by speculation */
    uint64_t spec_used;        /* missed experts read from the prefetch bank instead of the host store */
} moe_stats_t;

typedef struct {
    int32_t num_pools, slots_per_pool;
    uint64_t slot_bytes, slot_stride, record_bytes;
    uint64_t pool_device_bytes;   /* slot pool(s) in HBM */
    uint64_t store_host_bytes;    /* pinned host store, every expert of every layer */
    uint64_t scratch_device_bytes;
    uint64_t fused_decode_calls;  /* decode calls launched as one kernel */
    uint64_t split_decode_calls;  /* decode calls launched as route, gate/up, down kernels */
} moe_info_t;

typedef struct moe_cache moe_cache_t;

/* Creates a handle: validates cfg, allocates the pinned host store that holds
 * every expert of every layer [PAGED, "What does Paged Experts actually do?"],
 * the slot pool(s) in device memory, the device slot tables (all slots empty,
 * LRU order 0..K-1) and scratch. expert_host, if not NULL, is [L] host
 * pointers each to E canonical records back to back; shared_host, if not NULL
 * and has_shared, is [L] host pointers to one canonical record each. Records
 * are copied and repacked; the caller may free them after return. Experts can
 * also be supplied later with moe_cache_load_experts / moe_cache_load_shared.
 * Errors: MOE_ERR_INVALID (shape, format or mode), MOE_ERR_CAPACITY (fewer
 * slots than top_k in a pool), MOE_ERR_OOM, MOE_ERR_CUDA. *out is NULL on
 * failure. */
moe_status_t moe_cache_create(const moe_config_t* cfg, const void* const* expert_host,
                              const void* const* shared_host, moe_cache_t** out);

/* Copies `count` canonical records (host, back to back) for experts
 * first..first+count-1 of `layer` into the pinned store, repacking them.
 * Synchronous; uses several host threads. MOE_ERR_INVALID on a bad range. */
moe_status_t moe_cache_load_experts(moe_cache_t* h, int32_t layer, int32_t first, int32_t count,
                                    const void* records);

/* Uploads the shared expert of `layer` (one canonical record, host) to its
 * resident device buffer. Synchronous. MOE_ERR_INVALID without has_shared. */
moe_status_t moe_cache_load_shared(moe_cache_t* h, int32_t layer, const void* record);

/* One MoE layer for T tokens, asynchronous on `stream` (a cudaStream_t, or
 * NULL for the legacy default stream):
 *   logits = hidden x router_w^T (+ router_bias); top-k with ties to the lower
 *   expert id; weights = softmax over the picks (norm_topk) or the full
 *   softmax read at the picks; the experts' slots are looked up, misses are
 *   uploaded into least-recently-used slots [EXPLAINER, "Inside llama.cpp PR
 *   #29887"]; out[t] = sum_j w[t,j] * down(silu(gate x) * up x) over the
 *   picks in rank order, plus the shared expert with weight 1.
 *   hidden    : device bf16 [T x H], row-major
 *   router_w  : device bf16 [E x H], row-major
 *   router_bias: device fp32 [E] or NULL
 *   out       : device fp32 [T x H]
 * T <= max_cache_tokens runs the cache transaction (decode). Larger T (prefill)
 * reads resident experts in place without changing the LRU order and stages
 * the others through a double-buffered arena in groups of prefill_group
 * [T4, "What the MoE Cache Actually Caches"; NVME, "Workflow"; FP4LOCAL,
 * "Prefill"]. For Q4_0, block-FP8 and NVFP4 experts the prefill FFN runs as
 * tensor-core grouped GEMMs with fp16 operands (Q4_0 and block-FP8 weights
 * are rounded to fp16 there; NVFP4 weights are exact) and the staging copies
 * run on an internal side stream beside them; every kernel of the call that
 * reads a staged group waits for its copy on `stream`, so work issued on
 * `stream` after the call is ordered after all of it.
 * Errors (nothing is enqueued and the state is untouched):
 * MOE_ERR_INVALID for a bad layer, T <= 0 or T > max_tokens, null pointers;
 * MOE_ERR_CAPACITY when T * top_k exceeds the layer's pool on the decode path
 * (the single-wave rule of [PAGED, "What happens with more than one
 * request?"]) and multi_wave is 0; with multi_wave 1 such a call runs as
 * waves of floor(slots / top_k) tokens, each with its own page-in, as that
 * section describes for batches past the rule. MOE_ERR_STATE if experts were
 * never loaded; MOE_ERR_CUDA if a launch fails. In MOE_UPLOAD_MEMCPY mode the
 * call synchronises `stream`. */
moe_status_t moe_layer_forward(moe_cache_t* h, const void* hidden, int32_t T, const void* router_w,
                               const float* router_bias, int32_t layer_id, float* out, void* stream);

/* Registers the router of `layer` for speculative routing (speculate = 1):
 * router_w device bf16 [E x H], router_bias device fp32 [E] or NULL, the
 * same buffers the caller passes to moe_layer_forward for that layer. The
 * caller keeps them alive and unchanged until it registers others or
 * destroys the handle; router_w NULL unregisters the layer. Speculation for
 * layer l + 1 runs only while its router is registered [NVME, "Workflow":
 * run the next layer's router on the current layer's input].
 * The side stream's work for layer l + 1 is ordered before layer l + 1's
 * expert kernels (and before any other layer's call) on the caller's stream,
 * so a stream that issues the layers in order, up to the last, holds no
 * side-stream work afterwards. MOE_ERR_INVALID for a bad layer. */
moe_status_t moe_cache_set_router(moe_cache_t* h, int32_t layer, const void* router_w, const float* router_bias);

/* Synchronises the device and copies the counters out. Returns
 * MOE_ERR_TIMEOUT (counters still copied) if a grid barrier of the one-kernel
 * decode path gave up waiting since the last reset: every CTA of that kernel
 * must be resident at once, which another workload holding SMs for over
 * 0.2 s can prevent; the handle's state is then suspect until
 * moe_cache_reset. */
moe_status_t moe_cache_stats(moe_cache_t* h, moe_stats_t* out);

/* Sizes and layout facts of the handle (host only, no sync). */
moe_status_t moe_cache_info(moe_cache_t* h, moe_info_t* out);

/* Records every subsequent forward (up to `capacity_calls`, ring buffer) in a
 * device trace; capacity 0 turns tracing off. */
moe_status_t moe_cache_trace_enable(moe_cache_t* h, int32_t capacity_calls);

/* Synchronises and copies the oldest-first trace into buf (host int32) as
 * consecutive records [layer, T, n_ids, n_hit, n_fill, n_uniq, ids[n_ids],
 * slot_of[n_ids], hit_of[n_ids], fill_expert[n_fill], fill_slot[n_fill]] where
 * ids are in [token][rank] order. *n_words receives the words written;
 * *n_records the records. The trace is cleared. MOE_ERR_INVALID if buf_words
 * is too small for the records held. */
moe_status_t moe_cache_trace_read(moe_cache_t* h, int32_t* buf, int64_t buf_words, int64_t* n_words,
                                  int32_t* n_records);

/* Synchronises and copies the number of slots each pool holds now into
 * sizes [pools] (host int32): slots_per_layer (or the shared pool's slots)
 * unless the per-layer capacity adapts. */
moe_status_t moe_cache_pool_slots(moe_cache_t* h, int32_t* sizes);

/* Synchronises and copies the cache state: slot_map [L x E] (slot or -1),
 * key_of [pools x K] (layer*E + expert or -1), order [pools x K] (slots from
 * least to most recently used). Any pointer may be NULL. */
moe_status_t moe_cache_get_state(moe_cache_t* h, int32_t* slot_map, int32_t* key_of, int32_t* order);

/* Synchronises and copies `bytes` of slot `slot` of pool `pool` (device) into
 * dst (host), and, if store_dst is not NULL, the same bytes of the pinned store
 * record of (layer, expert) held there, for byte-exact upload checks. */
moe_status_t moe_cache_read_slot(moe_cache_t* h, int32_t pool, int32_t slot, void* dst,
                                 int32_t layer, int32_t expert, void* store_dst, uint64_t bytes);

/* Per-stage device timing for measurement: when enabled, every kernel a
 * forward launches is bracketed by CUDA events on the forward's stream (do
 * not enable it while capturing a CUDA graph). Stages: 0 router + top-k +
 * plan, 1 miss copies, 2 gate/up + SwiGLU, 3 down + combine, 4 prefill top-k,
 * 5 prefill plan, 6 the whole decode call in one kernel. */
#define MOE_NUM_STAGES 7
typedef struct {
    double ms[MOE_NUM_STAGES];         /* summed event time per stage */
    uint64_t launches[MOE_NUM_STAGES]; /* kernels timed per stage */
} moe_profile_t;

moe_status_t moe_cache_profile_enable(moe_cache_t* h, int32_t on);

/* Synchronises, returns the totals since the last read and clears them. */
moe_status_t moe_cache_profile_read(moe_cache_t* h, moe_profile_t* out);

/* Router + top-k of one layer that allocates nothing (no counterpart on the
 * pages: it exists for callers of this library that cannot call cudaMalloc
 * where they route tokens -- custom allocators that must not be re-entered
 * from their own callbacks, embedders that budget all device memory up front,
 * and latency-critical loops that cannot take cudaMalloc's implicit device
 * synchronisation). Computes, for T tokens, the same
 * routing as moe_layer_forward: logits = hidden x router_w^T (+ bias), the
 * top_k experts with ties to the lower id, and their weights (softmax over the
 * picks when norm_topk, else the full softmax read at the picks).
 *   hidden      : device bf16 [T x hidden_size]
 *   router_w    : device bf16 [num_experts x hidden_size]
 *   router_bias : device fp32 [num_experts] or NULL
 *   ids         : device int32 [T x top_k] (output, rank order per token)
 *   weights     : device fp32 [T x top_k] (output)
 * Limits: T <= 32, num_experts <= 512, top_k <= 16, hidden_size a multiple of
 * 64 up to 4096 (any such size: the router reads 256-column rounds and the last
 * one may be partial); anything else returns MOE_ERR_INVALID without launching.
 * Scratch: a fixed 196,864-byte array inside the library, held by every GPU
 * that loads it until the process exits; no call allocates or frees memory.
 * The first call on a device looks up the array's device address (make that
 * call before any stream capture); every later call only enqueues a memset of
 * an internal counter and one kernel on `stream`. All calls on a device share
 * the array, so calls whose kernels overlap on the GPU (unordered streams)
 * race. Asynchronous; MOE_ERR_CUDA if a launch fails. */
moe_status_t moe_route_topk_noalloc(const void* hidden, int32_t T, const void* router_w, const float* router_bias,
                                    int32_t num_experts, int32_t hidden_size, int32_t top_k, int32_t norm_topk,
                                    int32_t* ids, float* weights, void* stream);

/* Synchronises, empties every slot, restores the initial LRU order and clears
 * the counters and trace. Expert data stays loaded. */
moe_status_t moe_cache_reset(moe_cache_t* h);

/* Synchronises and frees everything the handle owns. NULL is accepted. */
moe_status_t moe_cache_destroy(moe_cache_t* h);

/* Last error message of the handle (or of the calling thread's last failed
 * create when h is NULL). Never NULL; valid until the next call on h. */
const char* moe_last_error(const moe_cache_t* h);

/* MOE_ABI_VERSION of the loaded library. */
int32_t moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_CACHE_H */
