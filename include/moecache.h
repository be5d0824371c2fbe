/*
 * moecache.h — C ABI of the bounded-expert-cache MoE layer for GB300 (sm_103a).
 *
 * One routed Mixture-of-Experts FFN layer whose quantised expert weights live
 * in a bounded cache of expert slots reached through a device page table:
 * router logits + top-k, expert-major union, cache resolve (admit / evict),
 * miss staging in 256 KiB tiles, fused dequantise + SwiGLU expert FFN with a
 * shared expert, and the weighted combine.
 *
 * Sources (page title and section):
 *   [MF]  "MawForge: Memory-Bounded Expert Materialization for Local MoE
 *         Inference", §IV-B split packs, §IV-C per-layer slot tensors and
 *         materialisation of misses, §IV-D static budget.
 *   [NfE] "Nanite for Experts", §1 model shape, §3.1 authoritative routing,
 *         §3.2 fail-closed correctness, §3.4 pinned host memory and
 *         non-default streams, §5.3 expert-major union, §5.4 256 KiB tiles,
 *         three streams and the persistent page table, §5.5 merge into
 *         original positions, §12 persistent expert-major operator.
 *   [RT]  "Paging the Experts" (Routide), §3.1 gate/up/down projections,
 *         §3.2 byte-budgeted cache with entries pinned per layer, §4.1/§5.1
 *         LRU versus seeded random eviction, §4.2 materialised-byte counters.
 *
 * Conventions
 *   - Every call returns moe_status_t; nothing throws across the ABI.
 *     moe_last_error(ctx) describes the last failure on that context.
 *   - Device pointers passed in are BORROWED: the caller owns and frees them
 *     and keeps them alive until the stream work that uses them has finished.
 *     The library owns the slot pools, page tables, generation arrays,
 *     scratch buffers, random-eviction state and its internal streams.
 *   - Stream arguments are cudaStream_t values (NULL = legacy default stream).
 *     Calls are stream-ordered and do not synchronise unless stated.
 *   - Layouts are row-major and dense. Expert payloads use the split-plane
 *     layout: for gate [I,H], up [I,H], down [H,I] in that order, a quant plane
 *     (Q8_0: int8 [rows][K]; Q4_0: uint8 [rows][K/2], byte j of a 32-block
 *     holds element j in its low nibble and element j+16 in its high nibble)
 *     followed by a little-endian fp16 scale plane [rows][K/32]. A weight is
 *     d*q (Q8_0) or d*(q-8) (Q4_0). All sizes K are multiples of 32. The
 *     affine INT4 format (MOE_I4_G64, below) keeps the same plane sizes.
 *   - A context is not thread-safe; use one per host thread.
 */
#ifndef MOECACHE_H
#define MOECACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* == cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,         /* invalid argument, size or pointer */
  MOE_ERR_CUDA = 2,        /* a CUDA runtime call failed */
  MOE_ERR_CAPACITY = 3,    /* the slots cannot hold what the step pins */
  MOE_ERR_STALE = 4,       /* a page-table entry or slot generation was invalid */
  MOE_ERR_TIMEOUT = 5,     /* a bounded device wait ran out */
  MOE_ERR_UNCERTIFIED = 6, /* routing could not be decided exactly */
  MOE_ERR_STATE = 7        /* call order violated (e.g. no store bound) */
} moe_status_t;

/* MOE_I4_G64: affine INT4 in groups of 64 along K ([RT] §3.1 gate/up/down
 * with scales and biases, BF16 quantisation metadata): x = s*q + b, q an
 * unsigned nibble, byte j of a row holding elements 2j (low nibble) and
 * 2j+1 (high nibble); the metadata plane holds the bf16 (s, b) pairs
 * [rows][K/64][2], as many bytes as a Q4_0 scale plane. Decode path only;
 * every K a multiple of 64. */
typedef enum { MOE_Q8_0 = 0, MOE_Q4_0 = 1, MOE_I4_G64 = 2 } moe_quant_t;
/* Policies of a context: LRU and seeded random. The other two exist for
 * offline replays only (moe_replay): farthest next use needs the future
 * route trace, and the static working set is a fixed resident set. */
typedef enum { MOE_LRU = 0, MOE_RANDOM = 1, MOE_FARTHEST_NEXT_USE = 2, MOE_STATIC_SET = 3 } moe_policy_t;
typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;
typedef enum { MOE_MODE_AUTO = 0, MOE_MODE_DECODE = 1, MOE_MODE_PREFILL = 2 } moe_mode_t;

/* Layer geometry and cache policy ([MF] §IV-C, [NfE] §1, [RT] §3.2). */
typedef struct {
  int32_t n_layers;        /* layers with their own slot pool */
  int32_t n_experts;       /* E routed experts per layer (<= 1024) */
  int32_t top_k;           /* k experts per token (<= 16) */
  int32_t hidden;          /* H (multiple of 32) */
  int32_t inter;           /* I, routed expert intermediate size (multiple of 32) */
  int32_t shared_inter;    /* I_s of the shared expert; 0 = no shared expert */
  int32_t quant;           /* moe_quant_t of every expert */
  int32_t slots_per_layer; /* S (1..n_experts) */
  int32_t policy;          /* moe_policy_t */
  int32_t n_streams;       /* staging streams (1..8; 3 in [NfE] §5.4) */
  uint64_t seed;           /* random-eviction seed */
  int64_t tile_bytes;      /* staging tile size, multiple of 16 (262144 in [NfE] §5.4) */
  int32_t max_tokens;      /* largest T of any call on this context */
  int32_t admit_on_device; /* 0: host slot manager, tiles staged on n_streams
                                 copy streams (admit syncs the stream);
                              1: admission on the GPU, misses staged by a copy
                                 kernel over the host link, no host sync;
                              2: admission on the GPU, misses materialised by
                                 the FFN while it reads them from the store */
  int32_t decode_ffn;      /* decode FFN (T <= 8): 0: two launches, gate/up
                                 then down (the default); 1: one persistent
                                 cooperative launch in which a read-through
                                 miss's down plane is copied into its slot in
                                 staging tiles, each with a ready counter that
                                 the down rows it holds wait on (bounded) */
} moe_config_t;

/* Expert-major plan ([NfE] §5.3, §5.5). Device arrays owned by the caller.
 * Assignment a = t*k + j is token t's j-th choice. The plan lists, for each
 * expert in ascending id, its assignments by ascending token. */
typedef struct {
  int32_t* counts;    /* [E] assignments per expert */
  int32_t* offsets;   /* [E+1] exclusive scan of counts */
  int32_t* uniq;      /* [E] experts with counts > 0, ascending; first n_uniq valid */
  int32_t* n_uniq;    /* [1] */
  int32_t* perm_tok;  /* [T*k] token of the p-th expert-major assignment */
  int32_t* perm_rank; /* [T*k] its rank j within the token's selection */
  float* perm_w;      /* [T*k] its combine weight */
  int32_t* inv;       /* [T*k] inv[t*k+j] = p */
  int32_t capacity;   /* assignments the arrays can hold (>= T*k) */
} moe_plan_t;

/* Fills decided by one cache resolve. Host arrays owned by the library,
 * valid until the next admit on the same context. */
typedef struct {
  int32_t n;              /* number of fills (= misses) */
  const int32_t* expert;  /* [n] expert materialised */
  const int32_t* slot;    /* [n] slot it goes to */
  const int32_t* victim;  /* [n] expert evicted from that slot, or -1 */
  const int32_t* wave;    /* [n] compute wave of the fill (0 unless |U| > S) */
  int32_t n_waves;        /* compute waves of the step (1 unless |U| > S) */
  int32_t hits;           /* assignments served by resident experts */
  int32_t misses;         /* experts materialised */
  int32_t layer;          /* layer the list belongs to */
} moe_miss_list_t;

typedef struct {
  int64_t steps;               /* cache resolves */
  int64_t hits;                /* assignment hits */
  int64_t misses;              /* expert misses */
  int64_t evictions;           /* slots reclaimed from a resident expert */
  int64_t materialized_bytes;  /* misses x payload ([RT] §4.2) */
  int64_t tiles_staged;        /* copy tiles issued by moe_stage_tiles */
  int64_t bytes_staged;        /* bytes copied by moe_stage_tiles */
  int64_t uncertified_repairs; /* tokens whose top-k needed exact logits */
  /* Confidence-gated prefetch ([RT] §3.3, §5.2), counted apart from the
   * demand counters above ([RT] §4.2): */
  int64_t prefetch_loads;      /* absent predicted experts loaded before their step */
  int64_t prefetch_useful;     /* loads whose next step's union held the expert */
  int64_t prefetch_wasted;     /* loads whose next step's union did not */
  int64_t prefetch_refreshes;  /* resident predictions touched like a hit */
  int64_t prefetch_probes;     /* resident predictions recorded, state unchanged */
  int64_t prefetch_bytes;      /* loads x payload */
  /* Many-token routing with the tensor-core filter: tokens whose certified
   * logit of a candidate fell outside the filter's interval, so that every
   * expert was taken as a candidate (the filter's error model failed; 0 is
   * expected, and the routing stays exact either way). */
  int64_t route_filter_fallbacks;
} moe_stats_t;

/* Prefetch modes ([RT] §3.3): an absent predicted expert is loaded in both;
 * a resident one is touched like a hit (RESIDENT_REFRESH: the check
 * updates its recency) or only recorded (PRESERVE: no state change). */
typedef enum { MOE_PREFETCH_OFF = 0, MOE_PREFETCH_REFRESH = 1, MOE_PREFETCH_PRESERVE = 2 } moe_prefetch_mode_t;
/* What one prefetch did. */
typedef enum { MOE_PREFETCH_PROBED = 0, MOE_PREFETCH_REFRESHED = 1, MOE_PREFETCH_LOADED = 2 } moe_prefetch_action_t;

typedef struct moe_ctx moe_ctx_t;
typedef struct moe_slots moe_slots_t;

/* ---------------------------------------------------------------- context */

/* Create a context on the CURRENT CUDA device: allocates S slots per layer
 * (each one expert payload), the device page table pt[L][E] (slot or -1),
 * pt_gen[L][E] and slot generations gen[L][S], and scratch for max_tokens.
 * Errors: MOE_ERR_ARG on an invalid config, MOE_ERR_CUDA if allocation fails
 * (*out is then NULL). */
moe_status_t moe_create(const moe_config_t* cfg, moe_ctx_t** out);

/* Synchronise the library's streams and free everything the context owns. */
void moe_destroy(moe_ctx_t* ctx);

/* Message of the last failing call on ctx (or of the last moe_create when
 * ctx is NULL). Owned by the library; valid until the next call. */
const char* moe_last_error(const moe_ctx_t* ctx);

/* Bytes of one routed expert payload and of the shared expert payload. */
int64_t moe_payload_bytes(const moe_ctx_t* ctx);
int64_t moe_shared_payload_bytes(const moe_ctx_t* ctx);

/* Bind the backing store of routed experts: PINNED host memory holding
 * payload [L][E] in split-plane layout, borrowed for the context's lifetime
 * ([MF] §IV-B split packs stand-in; [NfE] §3.4 pinned host memory).
 * Binding reads one 32-bit word of every 4 KiB page of the store from the
 * device and waits for it (about 0.1 s for 34 GB), so that the first miss
 * on each page does not pay the device's first-access cost of host memory.
 * Errors: MOE_ERR_ARG if bytes != L*E*payload or the memory is not
 * page-locked; MOE_ERR_CUDA if that read fails. */
moe_status_t moe_bind_store(moe_ctx_t* ctx, const void* pinned_host_store, size_t bytes);

/* Bind the always-resident shared expert of a layer ([NfE] §1): a DEVICE
 * pointer to one shared payload, borrowed. Required before moe_expert_ffn
 * when shared_inter > 0. */
moe_status_t moe_bind_shared(moe_ctx_t* ctx, int32_t layer, const void* dev_shared_payload);

/* ---------------------------------------------------------------- hot path */

/* Router + top-k ([NfE] §3.1 authoritative routing; [RT] §3.1 top-eight).
 * x: device [T,H] (xt = MOE_F32 or MOE_BF16); w_router: device fp32 [E,H];
 * both 16-byte aligned (MOE_ERR_ARG otherwise); bias: device fp32 [E] or NULL. Writes topk_idx int32 [T,k] (descending
 * logit, ties to the lower id) and topk_w fp32 [T,k] (softmax over the k
 * selected logits). The selection equals the one made on the correctly
 * rounded exact logits sum_i x_i*w_i (+b): fast fp32-pair logits carry an
 * error bound and any token whose order the bound cannot certify is
 * recomputed exactly on the device. 1 <= T <= max_tokens. */
moe_status_t moe_route(moe_ctx_t* ctx, int32_t layer, const void* x, int32_t xt, int32_t T,
                       const float* w_router, const float* bias, int32_t* topk_idx,
                       float* topk_w, moe_stream_t stream);

/* Router + top-k that allocates nothing, for callers that cannot call
 * cudaMalloc: code running inside another framework's memory pool or arena,
 * services that forbid device allocation after start-up, or work being
 * captured into a CUDA graph, where an allocation would break the capture.
 * None of the pages has a counterpart to this call; it exists for such
 * embedders. It needs no context: the caller passes x (device [T,H],
 * MOE_F32 or MOE_BF16), w_router (device fp32 [E,H]), bias (device fp32 [E]
 * or NULL) and the outputs topk_idx (int32 [T,k]) and topk_w (fp32 [T,k]);
 * the selection and weights are those of moe_route.
 * Scratch: one static device array inside the library, sized for
 * T*E <= 8192 logits (about 192 KiB), which every GPU that loads the library
 * holds until the process exits. Limits: 1 <= T <= 64, H a multiple of 4,
 * 1 <= E <= 1024, 1 <= k <= min(16, E), T*E <= 8192, x and w_router 16-byte
 * aligned; anything else returns MOE_ERR_ARG with a message in
 * moe_last_error(NULL) and launches nothing.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture. The address is then kept per device ordinal for the life of the
 * process: after cudaDeviceReset on that device it no longer names the
 * array, so do not call this entry point on a device that has been reset. No call allocates (no cudaMalloc, cudaFree or allocating library
 * routine). Every call shares the one array: it clears its counters on the
 * stream before the launch, and calls whose kernels overlap on the GPU (on
 * different streams, or from several threads) race on it — serialise them.
 * Device-side flags (non-finite inputs) are not reported by this call. */
moe_status_t moe_route_noalloc(const void* x, int32_t xt, int32_t T, int32_t H, int32_t E,
                               int32_t k, const float* w_router, const float* bias,
                               int32_t* topk_idx, float* topk_w, moe_stream_t stream);

/* Expert-major union and permutation of a routed step ([NfE] §5.3, §5.5).
 * topk_idx/topk_w: device [T,k]. Fills every array of *plan (device).
 * Errors: MOE_ERR_ARG if plan->capacity < T*k. */
moe_status_t moe_plan_union(moe_ctx_t* ctx, const int32_t* topk_idx, const float* topk_w,
                            int32_t T, const moe_plan_t* plan, moe_stream_t stream);

/* Cache resolve of one layer step ([MF] §IV-C, [RT] §3.2, §4.1). Reads the
 * plan's union and counts (copies them to the host and SYNCHRONISES
 * stream), classifies hits and misses, picks victims (LRU or seeded random),
 * assigns slots, updates the host page table and enqueues its copy to the
 * device page table on stream. The miss list must be staged with
 * moe_stage_tiles before moe_expert_ffn reads the slots.
 * Errors: MOE_ERR_CAPACITY when the random policy has no unpinned victim, or
 * when the step's union is larger than the slots (such a step runs only
 * inside moe_layer_forward, in compute waves); the cache state is then
 * unchanged. */
moe_status_t moe_cache_admit(moe_ctx_t* ctx, int32_t layer, const moe_plan_t* plan,
                             moe_miss_list_t* misses, moe_stream_t stream);

/* Explicit eviction of one expert of a layer (host and device page table);
 * its slot becomes free. Not stream-ordered: synchronises the library's
 * streams first. No-op for an absent expert. */
moe_status_t moe_cache_evict(moe_ctx_t* ctx, int32_t layer, int32_t expert);

/* Fill slots with the given experts before the first step (not counted as
 * misses). Copies synchronously; used for all-resident runs. */
moe_status_t moe_cache_preload(moe_ctx_t* ctx, int32_t layer, const int32_t* experts, int32_t n);

/* Miss staging ([NfE] §5.4): copy every fill of *misses from the bound
 * pinned store into its slot. The payload is cut into tiles of at most
 * tile_bytes (each matrix separately, the last tile partial): the unit of
 * the tile counters and of the failure hook. The consecutive tiles of one
 * fill are issued as one copy, and fills rotate over the context's
 * n_streams streams. Then each slot's new generation is published. compute_stream
 * waits (cudaStreamWaitEvent) for all of it, so moe_expert_ffn enqueued on
 * compute_stream afterwards reads complete slots. Overwriting a slot waits
 * for the compute previously enqueued on compute_stream. */
moe_status_t moe_stage_tiles(moe_ctx_t* ctx, int32_t layer, const moe_miss_list_t* misses,
                             moe_stream_t compute_stream);

/* Fused dequantise + SwiGLU expert FFN + shared expert + weighted combine
 * ([RT] §3.1, [NfE] §1, §5.5, §12). x: device [T,H]; plan from
 * moe_plan_union on this step; y: device fp32 [T,H], overwritten with
 * sum_j w[t,j] * FFN_{idx[t,j]}(x[t]) + FFN_shared(x[t]); x and y 16-byte
 * aligned (else MOE_ERR_ARG). Experts are read
 * from their slots through the device page table; an absent expert or a
 * slot whose generation differs from the page table's is not read: the step
 * then fails closed (MOE_ERR_STALE from moe_check_device_errors) and y is
 * left unspecified. mode: MOE_MODE_DECODE (T <= 8, dequant-GEMV),
 * MOE_MODE_PREFILL (Q8_0 only, contexts with max_tokens > 8: grouped
 * dequant-GEMM on the tensor cores, H % 128 == 0, I and I_s multiples of
 * 64), AUTO picks by T. */
moe_status_t moe_expert_ffn(moe_ctx_t* ctx, int32_t layer, const void* x, int32_t xt, int32_t T,
                            const moe_plan_t* plan, float* y, int32_t mode, moe_stream_t stream);

/* route -> plan -> admit -> stage -> ffn for one layer step (one host sync,
 * inside admit). misses may be NULL.
 * Host admission, T > 8, LRU: a step whose union is larger than the slots
 * runs in compute waves ([RT] §3.2 read as textbook LRU over the access
 * sequence): a fill that evicts an expert of the same step belongs to the
 * wave after that expert's. The activations are gathered once; per wave the
 * wave's fills are staged (after the previous wave's GEMMs) and the grouped
 * GEMMs run over the wave's experts, in two parts: the resident experts and
 * first fills, then the last quarter of the fills, whose copies overlap the
 * first part's GEMMs (a wave's fills never evict its own experts). A copy
 * failure leaves the whole wave unpublished. One combine follows. The output is the
 * same, bit for bit, as with every expert resident. Decode (T <= 8) returns
 * MOE_ERR_CAPACITY for such a step; on-device admission admits nothing and
 * moe_check_device_errors reports MOE_ERR_CAPACITY. */
moe_status_t moe_layer_forward(moe_ctx_t* ctx, int32_t layer, const void* x, int32_t xt,
                               int32_t T, const float* w_router, const float* bias,
                               int32_t* topk_idx, float* topk_w, const moe_plan_t* plan,
                               float* y, moe_miss_list_t* misses, moe_stream_t stream);

/* Confidence-gated prefetch ([RT] §3.3; the page applies it during
 * prefill): with mode != MOE_PREFETCH_OFF, every moe_layer_forward of this
 * context first prefetches the layer's prediction from its previous step,
 * namely the rank-0 expert of that step's last token when its combine
 * weight is >= threshold (0.20 on the page). An absent expert is loaded
 * into a slot chosen as for a miss with nothing pinned (the lowest free
 * slot, else the policy's victim); its copy goes out on the staging streams
 * before the step's routing, so it overlaps the routing and the host
 * admission, and its generation is published once it has landed. Routing
 * and outputs do not change (cache transparency); hits, misses and victims
 * may. Counted in moe_stats_t.prefetch_*. Host admission only
 * (admit_on_device = 0): MOE_ERR_STATE otherwise; MOE_ERR_ARG for a bad
 * mode or a threshold outside [0, 1]. Clears every layer's prediction. */
moe_status_t moe_set_prefetch(moe_ctx_t* ctx, int32_t mode, float threshold);

/* Synchronise stream and report device-side failures recorded since the
 * last check (stale page-table entries, timed-out waits); clears them. */
moe_status_t moe_check_device_errors(moe_ctx_t* ctx, moe_stream_t stream);

/* ---------------------------------------------------------------- inspection */

/* Counters of one layer (layer = -1: summed over layers) ([MF] §IV-C
 * telemetry; [RT] §4.2). */
moe_status_t moe_get_stats(const moe_ctx_t* ctx, int32_t layer, moe_stats_t* out);

/* Copy the DEVICE page table of a layer to host_pt [E] (slot or -1) and the
 * device slot generations to host_gen [S]; synchronises the library's
 * streams. Either output may be NULL. */
moe_status_t moe_read_page_table(moe_ctx_t* ctx, int32_t layer, int32_t* host_pt,
                                 uint32_t* host_gen);

/* Copy the bytes held by one slot of a layer to host memory (bytes <=
 * payload). Synchronises. For tests of staging. */
moe_status_t moe_read_slot(moe_ctx_t* ctx, int32_t layer, int32_t slot, void* host_out,
                           size_t bytes);

/* Kernel timing (tracing aid). While enabled, the context records CUDA
 * events on the launching stream around every kernel it launches.
 * moe_get_kernel_times synchronises those events and returns, per kind
 * (route incl. fused plan and on-device admission, standalone plan, prefill
 * FFN gate/up, prefill FFN down, on-device staging copy, decode FFN: gate/up,
 * down and the misses' tiles in one launch), the summed device milliseconds
 * and the launch count since the last call, then resets them. Either output
 * may be NULL. */
typedef enum {
  MOE_KT_ROUTE = 0,
  MOE_KT_PLAN = 1,
  MOE_KT_GATEUP = 2,
  MOE_KT_DOWN = 3,
  MOE_KT_STAGE = 4,
  MOE_KT_FFN = 5,
  MOE_KT_COUNT = 6
} moe_kernel_kind_t;
moe_status_t moe_set_kernel_timing(moe_ctx_t* ctx, int32_t enable);
moe_status_t moe_get_kernel_times(moe_ctx_t* ctx, double* ms, int64_t* launches);

/* Test hooks for fail-closed paths, all on the host side: make host staging
 * (moe_stage_tiles, or a wave of moe_layer_forward) fail once
 * `fail_after_tiles` more tiles have been issued (-1 = off), or change
 * the published generation of the slot holding a resident expert so that it
 * no longer matches the page-table entry. */
moe_status_t moe_debug_fail_staging_after(moe_ctx_t* ctx, int32_t fail_after_tiles);
moe_status_t moe_debug_corrupt_generation(moe_ctx_t* ctx, int32_t layer, int32_t expert);

/* Test hook of the device's bounded waits ([NfE] §3.2 fail closed on a
 * deadline): the next prefill gate/up GEMM of this context (one launch; the
 * hook then clears itself) limits each of its mbarrier waits to
 * wait_cycles SM clock cycles (0: the default, about 2 s) and its first CTA
 * issues no copy for ring stage skip_ring (-1: off), so that no copy is in
 * flight for that stage and the consumers' wait on it runs out. The kernel
 * then raises its abort flag, drains the copies and MMAs it did issue,
 * frees its tensor memory and returns; moe_check_device_errors reports
 * MOE_ERR_TIMEOUT and the context stays usable. Host side only: no wait is
 * removed and nothing faults. */
moe_status_t moe_debug_prefill_wait_timeout(moe_ctx_t* ctx, int64_t wait_cycles, int32_t skip_ring);

/* ---------------------------------------------------------------- slot manager
 * The host-side policy of the cache on its own (no CUDA calls): the same
 * object each context keeps per layer. Usable without a GPU. */

/* Cache of S slots over E experts for one layer; payload_bytes feeds the
 * materialised-byte counter. seed/layer key the random policy's SplitMix64
 * stream (seed XOR layer*0x9E3779B97F4A7C15). */
moe_status_t moe_slots_create(int32_t n_experts, int32_t n_slots, int32_t policy, uint64_t seed,
                              int32_t layer, int64_t payload_bytes, moe_slots_t** out);
void moe_slots_destroy(moe_slots_t* s);

/* Resolve one step: uniq[n_uniq] distinct experts (any order), counts[E]
 * assignments per expert. Fills *out (arrays owned by s, valid until the
 * next call). Access order: resident experts ascending, then missing experts
 * ascending; a miss takes the lowest free slot, else a victim (LRU: oldest
 * access; RANDOM: cand[next() mod n] over resident experts not in uniq,
 * listed by slot). MOE_ERR_CAPACITY (state unchanged) when RANDOM has no
 * candidate. */
moe_status_t moe_slots_step(moe_slots_t* s, const int32_t* uniq, int32_t n_uniq,
                            const int32_t* counts, moe_miss_list_t* out);
/* Prefetch one expert before the next step ([RT] §3.3): mode
 * MOE_PREFETCH_REFRESH or MOE_PREFETCH_PRESERVE (see moe_set_prefetch).
 * *action receives a moe_prefetch_action_t; *fill the load (n = 1: expert,
 * slot, evicted expert or -1) or nothing (n = 0), arrays owned by s and
 * valid until the next call. The next moe_slots_step counts a load useful
 * or wasted. */
moe_status_t moe_slots_prefetch(moe_slots_t* s, int32_t expert, int32_t mode, int32_t* action,
                                moe_miss_list_t* fill);
moe_status_t moe_slots_preload(moe_slots_t* s, const int32_t* experts, int32_t n);
moe_status_t moe_slots_evict(moe_slots_t* s, int32_t expert);
/* pt [E] (slot or -1) and gen [S]; either may be NULL. */
moe_status_t moe_slots_read(const moe_slots_t* s, int32_t* pt, uint32_t* gen);
moe_status_t moe_slots_stats(const moe_slots_t* s, moe_stats_t* out);

/* Next output of SplitMix64 from state *state (advanced in place). */
uint64_t moe_splitmix64_next(uint64_t* state);

/* ---------------------------------------------------------------- replay
 * Offline replay of one layer's step sequence under a cache policy, for
 * comparing policies on a fixed route trace ([RT] §2 farthest-next-use as
 * the offline paging reference, §5.1 fixed replays; [NfE] §5.6, §7.4 a
 * learned static working set). Step t's union is experts[offsets[t] ..
 * offsets[t+1]) (distinct ids, any order) with counts[i] assignments of
 * experts[i]; the union is pinned during its step. MOE_LRU and MOE_RANDOM
 * behave as moe_slots_step (seed, layer). MOE_FARTHEST_NEXT_USE: a miss
 * (ascending id after the hits) takes the lowest free slot, else evicts the
 * resident expert outside the union whose next step of use is the farthest
 * (never again is farthest; ties to the lower slot). MOE_STATIC_SET: the
 * width experts with the most assignments over the first calib steps (ties
 * to the lower id) are resident before the first step and never evicted;
 * every other expert of a step is a miss that is not admitted. Fills *out
 * (steps, hits = assignments - misses, misses, evictions, materialised =
 * misses x payload_bytes). Host only. Errors: MOE_ERR_ARG for bad input,
 * MOE_ERR_CAPACITY when a union exceeds the slots (random, farthest next
 * use) or width exceeds them. */
moe_status_t moe_replay(int32_t policy, int32_t n_experts, int32_t n_slots, uint64_t seed, int32_t layer,
                        int64_t payload_bytes, int32_t width, int32_t calib, int32_t n_steps,
                        const int32_t* offsets, const int32_t* experts, const int32_t* counts,
                        moe_stats_t* out);

/* ---------------------------------------------------------------- budget
 * Static budget check before serving ([MF] §IV-D): the lower bound
 * L(p, n) = C + E(p) + K(n) of the footprint F(p, n) = L(p, n) + O, with C
 * the resident common tensor bytes, E(p) the expert-cache budget at cache
 * fraction p, K(n) the KV-cache bytes at context n and O the runtime
 * overhead. A row whose lower bound exceeds the serving target is rejected
 * (accepted = 0), which is a result, not an error. p is given in parts per
 * million; E(p) = floor(p * layers * experts * payload_bytes); the slots of
 * a layer are floor(p * experts); K(n) = kv_bytes_per_token * n. Host only,
 * no CUDA call. Errors: MOE_ERR_ARG for a negative input, p above 10^6 or a
 * byte count that overflows int64. */
typedef struct {
  int64_t common_bytes;    /* C */
  int64_t expert_bytes;    /* E(p) */
  int64_t kv_bytes;        /* K(n) */
  int64_t overhead_bytes;  /* O */
  int64_t lower_bound;     /* L(p, n) */
  int64_t footprint;       /* F(p, n) */
  int32_t slots_per_layer; /* floor(p * experts) */
  int32_t accepted;        /* 1 if L(p, n) <= target_bytes */
} moe_budget_t;
moe_status_t moe_static_budget(int32_t n_layers, int32_t n_experts, int64_t payload_bytes, int64_t cache_ppm,
                               int64_t common_bytes, int64_t kv_bytes_per_token, int64_t context,
                               int64_t overhead_bytes, int64_t target_bytes, moe_budget_t* out);

#ifdef __cplusplus
}
#endif
#endif /* MOECACHE_H */
