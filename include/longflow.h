/*
 * longflow.h -- C ABI of the LongFlow fused decode step on a static KV slab.
 *
 * The operation (one call = one layer, every sequence of the batch):
 *
 *   for every sequence b and KV head g, with the G = q_heads / kv_heads query
 *   heads h in g's group (query head h reads KV head floor(h / G)):
 *     s_{h,i}  = (q_h . k_i) / sqrt(d)   over the n cached slots i and the new token
 *     alpha    = softmax_i(s_{h,i})      (the new token attends to itself)
 *     out_h    = sum_i alpha_{h,i} v_i
 *       -- "LongFlow Guide: KV Cache Compression for Reasoning AI", section
 *          "Mathematical Derivation of the LongFlow Score", alpha_{t,i} and o_t;
 *     score_i  = ||v_i||_1 * sum_{h in group} alpha_{h,i}
 *       -- same section, Score_LongFlow(i) = ||c_{t,i}||_1 = alpha_{t,i} ||v_i||_1,
 *          and "LongFlow: Efficient KV Cache Compression for Reasoning M"
 *          (gist.science summary), section 2.1, LongFlowScore(t_i) = alpha_i^t ||v_i||_1;
 *     if n < budget_b:   the new token takes slot n           (initial fill)
 *     else:              victim e = argmin score_i over slots whose position is
 *                        older than the protected window (pos_i < p - window),
 *                        exact ties to the lowest slot; the new token's K, V,
 *                        ||v||_1 and position overwrite slot e in place
 *       -- guide, section "Static Memory Pre-Allocation and In-Place Eviction",
 *          steps 1-3; summary, section 2.3 "Static KV Cache" / "Fused Kernel".
 *
 * Policy variants (lf_config; the defaults are the operation above):
 *   norm = 2       score_i = ||v_i||_2 * sum_h alpha_{h,i}: the guide, same section,
 *                  lets the importance be either the l1 or the l2 norm of c_{t,i};
 *   sinks = s      positions 0..s-1 are never evicted (the guide's reference step,
 *                  section "End-to-End Implementation", protects its first
 *                  sink_size slots);
 *   deferred = 1   the order of that reference step and of the fused kernel's step 4,
 *                  whose output is the slot that the following step overwrites:
 *                  the new token first takes the next free slot, or
 *                  the slot chosen at the previous step, and is attended from the
 *                  buffer; once the buffer is full the lowest-score slot with
 *                  pos_i < p + 1 - window becomes the slot the next token takes
 *                  (window >= 1 protects the new token itself);
 *   scope = LF_SCOPE_LAYER  one victim per (layer, sequence) shared by all KV heads,
 *                  scored by the sum over every query head (the reference step sums
 *                  |c| over heads and feature dimensions);
 *   score = LF_SCORE_H2O    score_i = the attention mass slot i's token has received,
 *                  summed over the group's query heads and over every decode step
 *                  since it entered the buffer, its entry step included (prompt
 *                  tokens start at 0) -- the cumulative statistic the guide
 *                  attributes to H2O (section "The Long-Output Reasoning Crisis"
 *                  and H2O's row of the comparison table).
 *
 * Storage: one static slab per cache, allocated once by lf_cache_create*,
 * never grown, moved or compacted.  All per-step work is stream-ordered and
 * asynchronous: no call below synchronises the host except lf_cache_check,
 * lf_prefill_fill's upload of the host prompt lengths, and create/destroy.
 *
 * Threading: a cache may be used from any host thread, but calls touching the
 * same layer must be ordered by the caller (same stream, or events).  With
 * scope = LF_SCOPE_LAYER every lf_decode_step of a cache must be ordered: the
 * per-slot score scratch the selection reads is one layer's, reused by all.
 * Device: every call must run with the device that was current at create.
 *
 * Errors: functions return LF_OK (0) or a negative lf_status and set a
 * thread-local message (lf_last_error).  Conditions detected on the device
 * (non-finite inputs, corrupted state, an expired bounded wait) are OR-ed
 * into a per-cache error word read and cleared by lf_cache_check.  No kernel
 * traps or waits without a bound.
 */
#ifndef LONGFLOW_H_
#define LONGFLOW_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LF_ABI_VERSION 6

typedef struct lf_cache lf_cache; /* opaque; owns the slab */

/* A cudaStream_t passed as a plain pointer; NULL is the legacy default stream. */
typedef void* lf_stream_t;

typedef enum lf_status {
  LF_OK = 0,
  LF_ERR_ARG = -1,         /* invalid argument (shape, range, null pointer) */
  LF_ERR_OOM = -2,         /* device allocation failed */
  LF_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed */
  LF_ERR_DEVICE = -5,      /* lf_cache_check: the device error word was set */
  LF_ERR_UNSUPPORTED = -7  /* valid but not built (head_dim, group size, smem) */
} lf_status;

typedef enum lf_dtype { LF_BF16 = 0, LF_F32 = 1 } lf_dtype;

/* What makes room in the cache (lf_config.evict). */
typedef enum lf_evict {
  LF_EVICT_OFF = 0,       /* full KV: append until the capacity, then read only */
  LF_EVICT_LONGFLOW = 1,  /* LongFlow: every step past the budget evicts one slot */
  LF_EVICT_RKV = 2        /* R-KV: append into a staging buffer; lf_rkv_compress
                             brings the cache back to its budget */
} lf_evict;

/* Which decode kernel to build the cache for. */
typedef enum lf_kernel {
  LF_KERNEL_AUTO = 0,        /* tensor cores where supported and the layer fits their
                                launch shape (per-cluster item table), else CUDA cores */
  LF_KERNEL_SIMT = 1,        /* CUDA-core dot products (every dtype / head_dim) */
  LF_KERNEL_TENSOR_CORE = 2  /* tcgen05 MMAs: bf16, head_dim 128, group 1/2/4/8 */
} lf_kernel;

/* How slots are scored for eviction. */
typedef enum lf_score {
  LF_SCORE_LONGFLOW = 0, /* alpha_i * ||v_i|| over the current step's weights */
  LF_SCORE_H2O = 1       /* cumulative attention mass (one fp32 accumulator per slot) */
} lf_score;

/* Which heads share one eviction decision. */
typedef enum lf_scope {
  LF_SCOPE_KV_HEAD = 0, /* every KV head evicts its own slot (scores summed over its group) */
  LF_SCOPE_LAYER = 1    /* one slot per (layer, sequence), scores summed over all heads */
} lf_scope;

/* Bits of the device error word (lf_cache_check). */
#define LF_DEVERR_NONFINITE 1 /* a softmax max/denominator was not finite */
#define LF_DEVERR_STATE 2     /* no eviction candidate / count out of range */
#define LF_DEVERR_TIMEOUT 4   /* a bounded on-chip wait expired; step skipped.  After
                                 it the step's outputs and the cache's contents are
                                 unspecified: restore them (lf_cache_layout) or recreate
                                 the cache; lf_cache_check also resets the internal
                                 exchange counters of split launches */

typedef struct lf_config {
  int dtype;              /* LF_BF16 or LF_F32: type of q, K, V, k_new, v_new, out */
  int evict;              /* lf_evict: 1 LongFlow eviction; 0 full KV -- append until the
                             capacity, then read only (no scores, no writes); 2 R-KV */
  const int32_t* budgets; /* host [batch] per-sequence budgets (each <= capacity and
                             > window when evicting), or NULL: every budget = capacity */
  int cluster;            /* CTAs that split one KV head's slots (1,2,4,8,16); 0 = auto */
  int stages;             /* depth of the shared-memory staging ring (2..16); 0 = auto */
  int kernel;             /* lf_kernel; LF_KERNEL_AUTO by default */
  /* Policy variants (see the top of the file); 0 everywhere is the default method.
   * Ignored when evict = 0, except norm, which sets what vnorm holds. */
  int score;              /* lf_score */
  int norm;               /* 1 (or 0) = ||v||_1, 2 = ||v||_2 */
  int sinks;              /* >= 0; window + sinks < every budget */
  int deferred;           /* 0 = victim chosen and overwritten in the same step,
                             1 = chosen now, overwritten by the next token (window >= 1) */
  int scope;              /* lf_scope */
  /* R-KV (evict = LF_EVICT_RKV; 0 = the README's default): `capacity` is the
   * retained budget plus the staging buffer.  bf16, head_dim 128, capacity <= 4096,
   * rkv_alpha * (q_heads / kv_heads) <= 64, no per-sequence budgets. */
  int rkv_buffer;         /* staging slots B_buffer (128) */
  int rkv_alpha;          /* observation queries, always-kept newest tokens (8) */
  int rkv_beta;           /* near-duplicates kept among the most recent (1) */
  float rkv_lambda;       /* importance / redundancy trade-off in (0, 1] (0.1) */
  float rkv_tau;          /* key cosine at or above which tokens are near-duplicates,
                             in (0, 1] (0.9) */
} lf_config;

/*
 * Create a cache of `layers` independent layers for `batch` sequences with
 * kv_heads KV heads of dimension head_dim, q_heads query heads (a multiple of
 * kv_heads), `budget` slots per (layer, sequence, KV head) and a protected
 * window of the `window` most recent positions (0 <= window < budget).
 * Storage is bf16, eviction on, the default policy.  Returns NULL on error (see
 * lf_last_error).
 * Supported: head_dim in {16, 32, 64, 128}; q_heads / kv_heads in {1, 2, 4, 8}.
 */
lf_cache* lf_cache_create(int layers, int batch, int kv_heads, int q_heads, int head_dim,
                          int budget, int window);

/* Same with explicit dtype / eviction mode / ragged budgets / launch shape.
 * `capacity` is the slot count of every slab unit (the largest budget when
 * evicting; the full-KV length when not).  cfg may be NULL (bf16, evict, the
 * default policy).  The H2O score adds one fp32 per slot, the deferred mode one
 * int32 per unit and the layer scope a one-layer scratch of one fp32 per slot;
 * all are allocated here. */
lf_cache* lf_cache_create_ex(int layers, int batch, int kv_heads, int q_heads, int head_dim,
                             int capacity, int window, const lf_config* cfg);

/* Free the slab and the handle.  NULL is accepted (no-op).  Returns LF_OK. */
int lf_cache_destroy(lf_cache* cache);

/*
 * Initial fill of one layer (guide, "Static Memory Pre-Allocation and
 * In-Place Eviction", step 1): sequence b's first prompt_len[b] tokens take
 * slots 0..prompt_len[b]-1 with positions 0..prompt_len[b]-1; ||v||_1 (||v||_2
 * with norm 2) is computed in fp32 from the stored values; the occupied count
 * and the next position become prompt_len[b].  Slots past the prompt are
 * marked empty.  H2O accumulators start at 0; no deferred victim is chosen.
 *   k, v        device, [batch][kv_heads][max_prompt][head_dim], cache dtype,
 *               contiguous, 16-byte aligned, caller-owned
 *   prompt_len  HOST [batch], 0 <= prompt_len[b] <= max_prompt and <= that
 *               sequence's budget (capacity when eviction is off; below the
 *               budget in deferred mode, so that the step which fills the
 *               buffer chooses the first victim); longer prompts are fed
 *               through lf_decode_step by the caller
 * The host lengths are uploaded before the call returns.  Stream-ordered.
 */
int lf_prefill_fill(lf_cache* cache, int layer, const void* k, const void* v,
                    const int32_t* prompt_len, int max_prompt, lf_stream_t stream);

/*
 * One fused decode step of one layer for every sequence (see the top of the
 * file).  All buffers are caller-owned, contiguous device memory that must
 * stay valid until the stream reaches the call (q, k_new and v_new 16-byte
 * aligned):
 *   q             [batch][q_heads][head_dim]   cache dtype
 *   k_new, v_new  [batch][kv_heads][head_dim]  cache dtype (the token's stored values)
 *   out           [batch][q_heads][head_dim]   cache dtype (fp32 accumulation, RNE rounding)
 *   evicted_slot  [batch][kv_heads] int32: the slot whose token left the buffer this
 *                 step (and took the new token), or -1 in the fill phase and in
 *                 eviction-off mode
 * Asynchronous; no host synchronisation; allocates nothing; capturable in a
 * CUDA graph.  Returns LF_ERR_ARG / LF_ERR_CUDA on a bad call or launch.
 * With the layer scope a step is two launches (the attention kernel, then a
 * per-sequence selection of the shared victim).
 */
int lf_decode_step(lf_cache* cache, int layer, const void* q, const void* k_new,
                   const void* v_new, void* out, int32_t* evicted_slot, lf_stream_t stream);

/*
 * R-KV's compression step ("GitHub - Zefan-Cai/R-KV", section "Method", stages
 * 2-4) for one layer of an LF_EVICT_RKV cache: every (sequence, KV head) holding
 * more than budget = capacity - rkv_buffer tokens is cut back to the budget.
 *   importance  I_i = mean over the rkv_alpha observation queries q_obs and the
 *               head's query group of their softmax weight on token i (softmax
 *               over every cached token, scale 1/sqrt(d));
 *   redundancy  R_i = 1 if at least rkv_beta later tokens have key cosine
 *               >= rkv_tau with token i, else 0;
 *   Z_i = rkv_lambda I_i - (1 - rkv_lambda) R_i; the rkv_alpha latest tokens
 *   stay, then the highest Z (equal Z: the later token) up to the budget.
 * The slab stays static: kept buffer tokens move into the freed slots below the
 * budget, in slot order.  Call it when the buffer is full (decode steps on a
 * full slab do not store the token and raise LF_DEVERR_STATE).
 *   q_obs  device, [batch][rkv_alpha][q_heads][head_dim] bf16: the queries of
 *          the rkv_alpha latest decode steps, any order, caller-owned
 * Stream-ordered, asynchronous, allocates nothing.  LF_ERR_ARG if the cache is
 * not an R-KV cache.
 */
int lf_rkv_compress(lf_cache* cache, int layer, const void* q_obs, lf_stream_t stream);

/* Synchronise `stream`, read and clear the device error word.  *bits (may be
 * NULL) receives the LF_DEVERR_* bits.  Returns LF_ERR_DEVICE if any was set. */
int lf_cache_check(lf_cache* cache, lf_stream_t stream, int32_t* bits);

/* Device pointers and shape of the slab, for inspection, snapshots and
 * restores by the caller (stream-ordered with the caller's own copies).
 * Element (layer l, sequence b, KV head g, slot s) of k/v starts at
 * ((((l * batch + b) * kv_heads + g) * slot_stride + s) * head_dim); vnorm and
 * pos use the same index without head_dim; count / next_pos are indexed
 * [(l * batch + b) * kv_heads + g]; budget is [batch]. */
typedef struct lf_layout {
  int layers, batch, kv_heads, q_heads, head_dim;
  int capacity;     /* usable slots per unit */
  int slot_stride;  /* allocated slots per unit (capacity rounded up) */
  int window, dtype, evict;
  int cluster, stages; /* launch shape of lf_decode_step */
  int kernel;          /* LF_KERNEL_SIMT or LF_KERNEL_TENSOR_CORE */
  void* k;          /* cache dtype */
  void* v;          /* cache dtype */
  float* vnorm;     /* fp32 ||v||_1 (||v||_2 with norm 2) of each slot, written at insert */
  int32_t* pos;     /* token position of each slot, -1 when empty */
  int32_t* count;   /* occupied slots */
  int32_t* next_pos;/* position of the next token */
  int32_t* budget;  /* per-sequence budget */
  int32_t* err;     /* device error word */
  int score, norm, sinks, deferred, scope; /* the policy (lf_config) */
  float* acc;       /* LF_SCORE_H2O: fp32 attention mass per slot (same index as
                       vnorm), else NULL */
  int32_t* pending; /* deferred: the slot the next token takes, per unit (same index
                       as count; -1 = none chosen), else NULL */
  int rkv_buffer, rkv_alpha, rkv_beta; /* R-KV parameters (evict = LF_EVICT_RKV) */
  float rkv_lambda, rkv_tau;
  int split_units;  /* tensor-core kernel with planned launches possible (see
                       lf_launch_plan): its resident clusters nc; 0 when steps never
                       take a plan (the CUDA-core kernel, or more resident clusters
                       than a plan can describe) */
  int32_t* split_cnt; /* planned launches: [split_units][2] arrival counts of the two
                       exchanges through global memory of a shared unit, at the row
                       of its first inner cut (see lf_launch_plan).  Zero between
                       launches; lf_cache_check zeroes them after an expired wait.
                       NULL when split_units is 0 */
} lf_layout;

int lf_cache_layout(const lf_cache* cache, lf_layout* out);

/*
 * The launch plan of the next lf_decode_step of `layer` (tensor-core kernel).
 * (No counterpart on the pages: this reports how the work of a step is spread
 * over the GPU, for tests and tuning.)
 *
 * A launch runs nc = lf_layout.split_units resident clusters.  Without a plan
 * (return value 0) cluster j takes the whole units j, j + nc, j + 2 nc, ... of
 * the layer (unit u = sequence u / kv_heads, KV head u % kv_heads).  With a plan
 * (return value nc) cluster j takes the whole units j, j + nc, ... below
 * *rounds * nc and, before them, one contiguous range of the units from
 * *rounds * nc on (units in order, slots in order within a unit): from slot
 * cut_slot[j] of unit cut_unit[j] to where cluster j + 1 starts (cut nc is
 * (units, 0)).  A unit cut inside (cut_slot > 0) is shared by the clusters whose
 * ranges meet it; they exchange through global memory, and its last range runs
 * to its occupied count at launch time.  The host takes a plan when its cost
 * model says it balances the clusters better than whole units and every
 * sequence of the layer holds at least 2048 tokens by the host's count of
 * prompts, decode steps and compressions (the counts only steer the plan;
 * results never depend on it).
 *   rounds              host, may be NULL
 *   cut_unit, cut_slot  host [max_cuts], filled when a plan is returned (both
 *                       NULL: not filled)
 * Returns 0 or nc, or a negative lf_status (LF_ERR_ARG: bad layer, or arrays
 * shorter than nc + 1).  Reads host state only: no device work, no allocation.
 */
int lf_launch_plan(lf_cache* cache, int layer, int32_t* rounds, int32_t* cut_unit,
                   int32_t* cut_slot, int max_cuts);

/*
 * The planner behind lf_launch_plan on given occupancies, without a cache or a
 * GPU (no counterpart on the pages; for tests and tuning).  occupancy [units]
 * host: the occupied slots of units 0..units-1; cluster: CTAs per cluster;
 * clusters: resident clusters (<= 152); max_items: units one cluster may
 * visit.  Returns `clusters` and fills *rounds, cut_unit and cut_slot [clusters
 * + 1] as lf_launch_plan does when a plan is taken (whatever the occupancies,
 * without the 2048-token rule), 0 when whole units are the cheaper launch, or
 * LF_ERR_ARG.
 */
int lf_launch_plan_for(const int32_t* occupancy, int units, int cluster, int clusters,
                       int max_items, int32_t* rounds, int32_t* cut_unit, int32_t* cut_slot);

/*
 * Prefill without any device allocation.  (No counterpart on the pages: this
 * is an integration entry point, not part of the method.)
 *
 * For callers that cannot call cudaMalloc at the point where they prefill:
 * an engine that reserves all device memory up front and hands out slices of
 * its own pool, code running where an allocation's implicit device
 * synchronisation is not allowed, or a runtime without access to the CUDA
 * allocator.  Such a caller owns the slab itself and describes it with an
 * lf_layout (k, v, vnorm, pos, count, next_pos, and layers, batch, kv_heads,
 * head_dim, capacity, slot_stride, dtype, norm; acc and pending when not
 * NULL; the other fields are ignored), laid out exactly as lf_cache_layout
 * documents.  The operation, argument meaning
 * and error behaviour are those of lf_prefill_fill, except that prompt
 * lengths are checked against `capacity` (the caller keeps its budgets):
 * prompt_len[b] <= capacity, and <= capacity - 1 when `pending` is not NULL
 * (deferred mode).  A caller whose budgets are below the capacity keeps
 * prompt_len[b] <= budget, and <= budget - 1 in deferred mode, itself: a
 * deferred buffer filled to its budget by the prompt reaches its next step
 * without a chosen slot, and that step raises LF_DEVERR_STATE.
 *
 * The prompt lengths travel to the GPU through a fixed array compiled into
 * the library (LF_NOALLOC_MAX_BATCH int32 entries, held by every GPU that
 * loads the library until the process exits); batches larger than that are
 * rejected with LF_ERR_ARG.  The array is shared by every call on a device and
 * keeps the last call's contents (each call overwrites the entries it reads),
 * so calls whose work overlaps on the GPU (different streams, no ordering)
 * race on it.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  The address is looked up again after the
 * device's CUDA context was replaced (a cudaDeviceReset in the process): the
 * first call after the reset, too, should come before any stream capture.
 * Nothing is allocated: no cudaMalloc, no cudaFree, no allocating library
 * routine.
 */
#define LF_NOALLOC_MAX_BATCH 16384
int lf_prefill_fill_noalloc(const lf_layout* dst, int layer, const void* k, const void* v,
                            const int32_t* prompt_len, int max_prompt, lf_stream_t stream);

/* Message of the last failed call on this thread ("" if none). */
const char* lf_last_error(void);

/* lf_status of the last failed call on this thread (LF_OK if none).  The way to
 * learn why lf_cache_create / lf_cache_create_ex returned NULL: LF_ERR_ARG,
 * LF_ERR_UNSUPPORTED, LF_ERR_OOM (the slab does not fit in device memory) or
 * LF_ERR_CUDA.  It keeps its value until the next failure, or until one of
 * lf_cache_create*, lf_cache_destroy, lf_prefill_fill, lf_prefill_fill_noalloc,
 * lf_cache_check and lf_cache_layout resets it (with the message) on entry. */
int lf_last_status(void);

/* LF_ABI_VERSION of the loaded library. */
int lf_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LONGFLOW_H_ */
