/*
 * moeslot.h -- C ABI of the slot-cached MoE layer (GB300, sm_103a).
 *
 * One MoE layer forward whose expert weights sit partly in a fixed pool of
 * VRAM slots and partly in pinned host memory:
 *   route (logits, soft-biased top-k, softmax weights) -> permute into
 *   per-expert groups -> expert_cache_manage -> expert_cache_gather (or
 *   zero-return) -> grouped SwiGLU expert FFN -> weighted combine.
 *
 * Conventions for every entry point
 *   - Pointers named "device" must be device memory (or managed memory);
 *     "host store" pointers must be pinned host memory the GPU can address
 *     (cudaHostAlloc / torch pin_memory()).  The caller allocates and owns
 *     every buffer; the library allocates no memory.  It keeps only cached
 *     CUDA event handles for the two-stream layer forward.
 *   - bf16 tensors are passed as void* (IEEE bfloat16, little endian).
 *   - Every call only enqueues work on the given stream(s) and returns; the
 *     results are valid once that work has completed.  No call synchronises
 *     with the host.  A NULL stream is the legacy default stream.
 *   - Host-detectable argument errors return a negative moe_status before
 *     anything is enqueued.  Errors found on the device (an expert id out of
 *     range) are written as a nonzero code into the caller's device int32
 *     `dev_status` (which the caller zeroes), the offending item is skipped,
 *     and no kernel traps.
 *   - Slab layout for expert e (bf16, contiguous, 3*H*I elements):
 *       [ Wg (H x I) | Wu (H x I) | Wd (I x H) ]  each row-major, input-major,
 *     so g = x Wg, u = x Wu, h = silu(g) * u, y = h Wd.
 *   - Shape limits: H % 64 == 0, I % 32 == 0, 1 <= k <= 16, k <= E <= 1024,
 *     1 <= T, 1 <= S <= 4096.  Pointers read with 16-byte vectors must be
 *     16-byte aligned (slabs, pool, host store, y, workspace).
 */
#ifndef MOESLOT_H
#define MOESLOT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same handle as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_ARG = -1,                   /* null pointer, bad shape, bad enum */
  MOE_ERR_CAPACITY = -2,              /* step needs more slots than the pool has */
  MOE_ERR_ALIGN = -3,                 /* slab size or a pointer not a 16-byte multiple, workspace too small */
  MOE_ERR_NOT_DEVICE_ACCESSIBLE = -4, /* host store not addressable by the GPU */
  MOE_ERR_CUDA = -5,                  /* a CUDA runtime call failed */
  MOE_ERR_DEVICE_STATUS = -6,         /* reserved: a kernel reported a bad item */
  MOE_ERR_SCRATCH_LIMIT = -7          /* request larger than the fixed scratch of moe_expert_ffn_noalloc */
} moe_status;

typedef enum { MOE_POLICY_LRU = 0, MOE_POLICY_LFU = 1, MOE_POLICY_STATIC = 2 } moe_policy;
typedef enum { MOE_MODE_RESIDENT = 0, MOE_MODE_GATHER = 1, MOE_MODE_ZERO_RETURN = 2 } moe_mode;

/* Device status codes written into dev_status. */
#define MOE_DEV_BAD_EXPERT 1 /* an expert id outside [0, E) */
#define MOE_DEV_BAD_SLOT 2   /* a slot id outside [0, S) where a slot was required */
#define MOE_DEV_TIMEOUT 3    /* a kernel gave up waiting for its own asynchronous copies */
#define MOE_DEV_BAD_GROUPS 4 /* group offsets that do not add up to the routed rows (more tiles than rows) */

const char* moe_status_str(int status);

/*
 * Soft selection bias for one layer.
 * Source: "Nudge, don't cut" (PGO-SGB), section "The method in five lines":
 * bias[e] = max(cap, ln(b[e] / b_edge)) outside the hot set, 0 inside it;
 * the hot set is the n_hot brightest experts (ties: lower id), b_edge the
 * smallest brightness in it.  Evaluated in fp64, rounded to fp32; b[e] <= 0
 * gives cap.  Built once per layer, before serving (the page reads the
 * table once at startup).
 *   b     device fp32 [E], brightness (>= 0)
 *   bias  device fp32 [E], output
 * Errors: MOE_ERR_ARG if a pointer is NULL, E < 1, E > 1024 or n_hot not in [1, E].
 */
int moe_bias_table(const float* b, int E, int n_hot, float cap, float* bias, moe_stream_t stream);

/* Bias table modes ("Nudge, don't cut", introduction: "Hard mask: cold
 * experts can never be picked" vs a soft bias; and its comparison of the
 * graded bias with a flat one). */
#define MOE_BIAS_GRADED 0 /* cold: max(value, ln(b / b_edge)), as moe_bias_table with cap = value */
#define MOE_BIAS_FLAT 1   /* cold: value (one constant, e.g. -0.5) */
#define MOE_BIAS_HARD 2   /* cold: -inf, so a cold expert is never picked while k hot experts exist */

/*
 * The bias table in any of the three modes; hot experts get 0 in all of them.
 * Arguments and errors as moe_bias_table; MOE_ERR_ARG also for an unknown mode.
 */
int moe_bias_table_mode(const float* b, int E, int n_hot, int mode, float value, float* bias,
                        moe_stream_t stream);

/*
 * Router: logits, top-k by logit + bias (+ affinity), softmax weights over the picked k.
 * Source: "Nudge, don't cut" (PGO-SGB), "The method in five lines" (pick
 * top-k by logit + bias; weights are the router's own softmax over the k
 * picked, from the unbiased logits).
 *   x            device bf16 [T][H]
 *   w_router     device bf16 [H][E]
 *   logit_offset device fp32 [E] added to every logit after the sum, or NULL
 *   sel_bias     device fp32 [E] selection-only bias, or NULL
 *   e2s, affinity  live-cache affinity ("Nudge, don't cut", "Then Maya's own
 *                knob beat ours"): with e2s (device int32 [E], the cache's
 *                expert -> slot table) and affinity != 0, experts with
 *                e2s[e] >= 0 get `affinity` added to their selection score
 *                (after the bias, fp32).  NULL / 0 = off.
 *   logits       device fp32 [T][E] output (unbiased logits)
 *   scratch      device, moe_route_scratch_bytes(T, H, E) bytes (one fp32 [T][E]
 *                part per 128-row block), or NULL: with it the 128-row blocks
 *                are spread over more CTAs and the parts added in block order
 *                (the result is the same bit for bit)
 *   ids          device int32 [T][k] output, descending score, ties -> lower id
 *   w            device fp32 [T][k] output, sums to 1 per token
 * logit[t][e] is accumulated in fp32 in one fixed order: h is cut into
 * blocks of 128 rows, each block summed from 0 with fma in h order, and the
 * block sums added in block order; so ids are reproducible bit for bit.
 * Errors: MOE_ERR_ARG on NULL pointers or shapes out of range (H % 8 and
 * E % 8 must be 0); MOE_ERR_ALIGN if x or w_router is not 16-byte aligned.
 */
int moe_route(const void* x, const void* w_router, const float* logit_offset, const float* sel_bias,
              const int32_t* e2s, float affinity, int T, int H, int E, int k, float* logits, float* scratch,
              int32_t* ids, float* w, moe_stream_t stream);
size_t moe_route_scratch_bytes(int T, int H, int E);

/* Router flags for moe_route_ex. */
#define MOE_ROUTE_SIGMOID 1 /* GLM's sigmoid router ("Nudge, don't cut", "The same idea on GLM-5.3-Flash":
                               the bias is added after the sigmoid, in probability space) */
#define MOE_ROUTE_DAMPED 2  /* damped weights ("Qwen on Strata": selection-only against damped): the
                               bias also enters the weights */

/*
 * moe_route with a router variant (rflags = 0 is moe_route):
 *   MOE_ROUTE_SIGMOID  score = sigmoid(logit) + bias (+ affinity), picked as
 *                      above; w[j] = sigmoid(logit_j) / sum over the picked k.
 *                      sigmoid(l) = 1 / (1 + e(-l)) in fp32, with e() one fixed
 *                      sequence of IEEE fp32 operations (Cody-Waite reduction,
 *                      degree-7 Taylor polynomial, times 2^n; +inf above 88, 0
 *                      below -80), so the ids are reproducible bit for bit.
 *   MOE_ROUTE_DAMPED   softmax router; w = softmax over the picked k of
 *                      logit + sel_bias (affinity stays selection-only).
 * Errors: as moe_route; MOE_ERR_ARG for unknown flags or SIGMOID with DAMPED.
 */
int moe_route_ex(const void* x, const void* w_router, const float* logit_offset, const float* sel_bias,
                 const int32_t* e2s, float affinity, int rflags, int T, int H, int E, int k, float* logits,
                 float* scratch, int32_t* ids, float* w, moe_stream_t stream);

/*
 * Permute: group the n = T*k routing slots by expert.
 * Source: "Porting vllm-expert-cache to NVIDIA GPUs", "What this package
 * does" (the fused MoE kernel runs on grouped, slot-remapped ids).
 *   ids     device int32 [n] (flat t*k + j)
 *   count   device int32 [E]      tokens routed to each expert
 *   offset  device int32 [E + 1]  exclusive prefix of count; offset[E] = n
 *   rows    device int32 [n]      flat index at each grouped position; within
 *                                 an expert, ascending flat index (stable)
 *   pos     device int32 [n]      grouped position of each flat index
 *   act_e   device int32 [E]      experts with count > 0, ascending
 *   n_act   device int32 [1]      their number
 *   scratch device, moe_permute_scratch_bytes(n, E) bytes, or NULL: with it,
 *           n > 1024 is grouped by ceil(n/1024) CTAs (histogram, scan,
 *           scatter); without it by one CTA.  The result is the same.
 *   dev_status device int32 [1]   set to MOE_DEV_BAD_EXPERT on an id outside [0, E)
 * Errors: MOE_ERR_ARG on NULL pointers, n < 1 or E out of range.
 */
int moe_permute(const int32_t* ids, int n, int E, int32_t* count, int32_t* offset, int32_t* rows,
                int32_t* pos, int32_t* act_e, int32_t* n_act, int32_t* scratch, int32_t* dev_status,
                moe_stream_t stream);
size_t moe_permute_scratch_bytes(int n, int E);

/*
 * expert_cache_manage: update the slot cache for one step and emit the miss list.
 * Source: "Porting vllm-expert-cache to NVIDIA GPUs", "What this package does"
 * (victims are picked among slots this step does not need; a miss list is
 * emitted; ids are remapped to slot space), "Prove it is correct before
 * measuring" (fields: expert-to-slot table, cold map, slot contents,
 * priorities, miss list; deterministic, no atomics), "Measuring, without
 * fooling yourself" (a step is served from slots only when tokens x top_k <= slots).
 * One CTA, no atomics; the result does not depend on thread timing.
 *   ids       device int32 [n] routing ids of the step
 *   e2s       device int32 [E]  expert -> slot, -1 = cold (in/out)
 *   s2e       device int32 [S]  slot -> expert, -1 = empty (in/out)
 *   prio      device uint32 [S] policy priority (in/out)
 *   stamp     device uint32 [1] call counter, +1 per call (in/out)
 *   miss_e    device int32 [>= min(n, E)] missing experts, ascending id
 *   miss_s    device int32 [same]   slot each one goes to (-1 under STATIC)
 *   n_miss    device int32 [1]
 *   hit_e     device int32 [>= min(n, E)] needed experts already resident, ascending, or NULL
 *   n_hit     device int32 [1], or NULL (both or neither)
 *   sid       device int32 [n] slot of each routing id after the call, or NULL
 * Policies: LRU (prio = stamp on hit or load), LFU (prio += 1 once per call
 * on a hit, prio = 1 on load), STATIC (never evicts; misses are listed with
 * slot -1 and left for a zero-return pass).  Victim order: empty slots
 * (ascending), then ascending prio, then ascending slot; the i-th missing
 * expert takes the i-th victim.  Eviction sets e2s[old] = -1 (no write-back:
 * the host store stays authoritative).
 * Errors: MOE_ERR_CAPACITY if policy != STATIC, S < E and n > S;
 * MOE_ERR_ARG on NULL pointers or bad shapes/policy.
 */
int moe_cache_manage(const int32_t* ids, int n, int E, int S, int policy, int32_t* e2s, int32_t* s2e,
                     uint32_t* prio, uint32_t* stamp, int32_t* miss_e, int32_t* miss_s, int32_t* n_miss,
                     int32_t* hit_e, int32_t* n_hit, int32_t* sid, int32_t* dev_status, moe_stream_t stream);

/*
 * expert_cache_gather: copy each missing expert's slab from the host store into its slot.
 * Source: "Porting vllm-expert-cache to NVIDIA GPUs", "What this package does"
 * (copies the missing experts host-to-slot), "1. Kernels" (16-byte copy
 * unit), "Prove it is correct before measuring" (the device reads host
 * memory; per-expert slabs must stay 16-byte multiples).
 * The kernel reads pinned host memory directly, 16 bytes per access; the
 * number of misses is read on the device, so no host round trip is needed.
 *   host_slabs  pinned host bf16 [E][slab_bytes/2], GPU-addressable (read)
 *   pool        device [S][slab_bytes/2] (written for listed slots only)
 *   miss_e, miss_s, n_miss  device, as written by moe_cache_manage
 *   max_miss    host upper bound on *n_miss (sizes the grid)
 * Errors: MOE_ERR_ALIGN if slab_bytes or a base pointer is not a 16-byte
 * multiple; MOE_ERR_NOT_DEVICE_ACCESSIBLE if host_slabs is not addressable
 * by the current device; MOE_ERR_ARG otherwise.  A listed slot outside
 * [0, S) or expert outside [0, E) is skipped and flagged in dev_status.
 */
int moe_cache_gather(const void* host_slabs, void* pool, size_t slab_bytes, int E, int S,
                     const int32_t* miss_e, const int32_t* miss_s, const int32_t* n_miss, int max_miss,
                     int32_t* dev_status, moe_stream_t stream);

/*
 * Grouped SwiGLU expert FFN over a device-side list of experts.
 * Sources: "Porting vllm-expert-cache to NVIDIA GPUs", "What this package
 * does" (the expert GEMM runs on slot-remapped ids); "RTX 3060 runs a 35B
 * MoE with llama.cpp", chapter "Designing a fixed expert cache with
 * zero-return for missing experts" (a pass over the experts on the GPU and
 * a pass over the ones still in host memory).
 * For each expert e in list_e[0 .. *n_list) and each grouped position p in
 * [offset[e], offset[e+1]): token t = rows[p] / k,
 *   h = silu(x[t] Wg_e) * (x[t] Wu_e)  (fp32),   y[p] = h Wd_e  (fp32).
 * Weights of e are read from pool + e2s[e] * slab when e2s[e] >= 0, else
 * straight from host_slabs + e * slab (the zero-return second pass).  With
 * e2s == NULL expert e sits in slot e.  The pool holds S slots.  With
 * host_slabs == NULL every listed expert must be in the pool; the weight
 * tiles are then streamed through shared memory with tensor-map bulk copies.
 *   x          device bf16 [T][H]
 *   offset     device int32 [E + 1], rows device int32 [T*k] (moe_permute)
 *   list_e     device int32 [>= *n_list], n_list device int32 [1]
 *   max_list   host upper bound on *n_list
 *   y          device fp32 [T*k][H]; only rows of listed experts are written
 *   workspace  device scratch of moe_ffn_workspace_bytes(T, H, k, I) bytes (holds h)
 * Large groups (T*k >= 4096, weights in the pool) run as two tcgen05 grouped
 * GEMMs (M = 128 rows x N = 256 columns, fp32 accumulation in TMEM, bf16 h)
 * when the workspace holds the extra buffers; smaller ones stream the weight
 * tiles once per batch of <= 8 rows.
 * Errors: MOE_ERR_ARG on NULL pointers or bad shapes, MOE_ERR_ALIGN on
 * unaligned weight/output pointers or a workspace that is too small.
 */
int moe_expert_ffn(const void* x, int T, int H, int I, int k, int E, const int32_t* offset,
                   const int32_t* rows, const int32_t* list_e, const int32_t* n_list, int max_list,
                   const void* pool, int S, const int32_t* e2s, const void* host_slabs, float* y,
                   void* workspace, size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream);

/* Workspace of moe_expert_ffn: fp32 h [T*k][I]; for T*k >= 4096 also the
 * bf16 grouped rows of x [T*k][H] and bf16 h [T*k][I] of the tensor-core path. */
size_t moe_ffn_workspace_bytes(int T, int H, int k, int I);

/*
 * The grouped expert FFN for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a deployment variant of
 * moe_expert_ffn, not part of the method.
 *
 * Some callers cannot call cudaMalloc (or any allocator) where they run the
 * FFN, for example code running in a host callback, a plug-in that must not
 * touch its host's memory pool, or a runtime whose allocator is frozen after
 * start-up.  This variant takes no workspace: the intermediate h lives in one
 * fixed device array inside the library, MOE_FFN_NOALLOC_MAX_H fp32 values
 * (4 MiB) that every GPU which loads the library holds until the process
 * exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 * Arguments, outputs, argument checks and results are those of
 * moe_expert_ffn without the workspace: S is the pool's slot count, a slot
 * outside [0, S) found on the device sets MOE_DEV_BAD_SLOT and skips the
 * expert.  With host_slabs == NULL the weight tiles are streamed through
 * shared memory by tensor-map copies (the CUDA-core kernel that takes no
 * partial-sum buffers); with host_slabs the host-weights kernel runs.  h is
 * kept in fp32, so y can differ from moe_expert_ffn's tensor-core paths by
 * the rounding of h to bf16 there.
 *   - Limit: T * k * I <= MOE_FFN_NOALLOC_MAX_H, else MOE_ERR_SCRATCH_LIMIT
 *     is returned and nothing is enqueued.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the array and it keeps the last call's contents.
 *     Nothing in it needs to start at zero (each call writes every h row it
 *     reads), but calls that overlap on the GPU (other streams, other host
 *     threads) race on it: serialise them.
 */
#define MOE_FFN_NOALLOC_MAX_H (1u << 20)
int moe_expert_ffn_noalloc(const void* x, int T, int H, int I, int k, int E, const int32_t* offset,
                           const int32_t* rows, const int32_t* list_e, const int32_t* n_list, int max_list,
                           const void* pool, int S, const int32_t* e2s, const void* host_slabs, float* y,
                           int32_t* dev_status, moe_stream_t stream);

/*
 * Weighted scatter-combine back to token order.
 * Source: "RTX 3060 runs a 35B MoE with llama.cpp", chapters "Designing a
 * fixed expert cache with zero-return for missing experts" and "Fixing
 * scheduler order to improve performance" (two runs, then one add).
 *   out[t] = bf16( sum_{j=0..k-1} w[t][j] * y[pos[t*k+j]] ), fp32, j ascending.
 * With split != 0 a routing slot counts as resident when e2s[ids[t][j]] >= 0;
 * out_res / out_miss (fp32 [T][H]) get the two partial sums and
 * out = bf16(out_res + out_miss).
 *   y device fp32 [T*k][H]; w device fp32 [T][k]; pos device int32 [T*k]
 *   ids, e2s device int32 (split only; e2s has E entries); out device bf16 [T][H]
 * Errors: MOE_ERR_ARG on NULL pointers or bad shapes.
 */
int moe_combine(const float* y, const float* w, const int32_t* pos, const int32_t* ids, const int32_t* e2s,
                int T, int k, int H, int E, int split, void* out, float* out_res, float* out_miss,
                moe_stream_t stream);

/*
 * Optional per-kernel timing of moe_layer_forward (tracing).  `events` holds
 * `capacity` cudaEvent_t handles created by the caller with timing enabled.
 * The layer forward records one (start, end) pair around each kernel it
 * launches, on the stream that kernel runs on, in launch order, while pairs
 * remain; `used` (out) is the number of handles recorded and tags[i] (out)
 * the kernel class of pair i.  Recording events adds no synchronisation.
 */
enum {
  MOE_PROF_ROUTE = 0,
  MOE_PROF_PERMUTE = 1,
  MOE_PROF_MANAGE = 2,
  MOE_PROF_GATHER = 3,
  MOE_PROF_FFN_GATEUP = 4,
  MOE_PROF_FFN_DOWN = 5,
  MOE_PROF_COMBINE = 6,
  MOE_PROF_FFN_ROWS = 7, /* grouped copy of the routed rows of x (tensor-core path) */
  MOE_PROF_DECODE = 8,   /* a persistent decode kernel (bf16 or W8A8): the whole layer in one launch */
  MOE_PROF_CLASSES = 9
};
typedef struct moe_prof {
  void** events;    /* cudaEvent_t[capacity] */
  int32_t capacity;
  int32_t used;     /* out */
  int32_t* tags;    /* [capacity / 2] out */
} moe_prof;

/*
 * Periodic re-pick of a STATIC pool.
 * Source: "RTX 3060 runs a 35B MoE with llama.cpp" (video transcript),
 * chapter on code and chat profiles: the static hot set is chosen once, yet
 * the useful set drifts; every few hundred tokens, have another look, swap
 * out whatever has gone cold and leave it alone again (transfers are paid
 * once per window, not per token).
 *
 * moe_cache_count adds one to counts[e] for every routing id e (device int32
 * [n] ids, device int32 [E] counts, both caller-owned; ids out of range set
 * MOE_DEV_BAD_EXPERT in dev_status and are skipped).
 *
 * moe_cache_repick keeps the S experts ranked first by (counts desc, resident
 * before cold, id asc).  New members (ascending id) take the empty slots
 * first, then the slots of experts that left the set (ascending slot); e2s and
 * s2e are updated, the loads are written as miss_e / miss_s (device int32 >=
 * min(S, E) entries) with their count in n_miss (device int32), and the counts
 * are cleared.  Priorities and stamp are untouched (the pool stays STATIC).
 * Copy the new members with moe_cache_gather on the same lists.
 * Errors: MOE_ERR_ARG on NULL pointers, E not in [1, 1024], S not in [1, 4096].
 */
int moe_cache_count(const int32_t* ids, int n, int E, int32_t* counts, int32_t* dev_status, moe_stream_t stream);
int moe_cache_repick(int32_t* counts, int E, int S, int32_t* e2s, int32_t* s2e, int32_t* miss_e, int32_t* miss_s,
                     int32_t* n_miss, moe_stream_t stream);

/*
 * W8A8 experts (8-bit weights and activations).
 * Source: "Porting vllm-expert-cache to NVIDIA GPUs": the measured model is
 * Qwen3-30B-A3B W8A8, and weights and their scales are indexed by the same
 * id, so both must be slot-indexed (section on traps in a new backend).
 *
 * Quantised slab, moe_q8_slab_bytes(H, I) = 3HI + 4(2I + H) bytes:
 *   Wg, Wu [H][I] and Wd [I][H] as int8, each column's 4 consecutive input
 *   rows packed into one 32-bit word (byte (k, n) at ((k/4)*N + n)*4 + k%4),
 *   then the fp32 scales sg[I], su[I], sd[H].  The scales travel with the
 *   weights: manage and gather (slab_bytes = moe_q8_slab_bytes) keep them in
 *   the same slot.
 * Codes: symmetric, scale = amax / 127, code = rint(v / scale) clamped to
 * [-127, 127] (a zero amax gives scale 0 and code 0), fp32 one operation at a
 * time.  Weights per output column; activations per routing row: x before
 * gate/up, h before down.  Dot products are exact int32 sums;
 * g = (float(acc) * sg[n]) * sx[row] (likewise u and y), h = silu(g) * u with
 * silu(g) = g / (1 + e(-g)) and e() the fp32 exp of moe_route_ex; so h's codes
 * and y are reproducible bit for bit.
 *
 * moe_quantize_slabs: src device bf16 [n_experts][3HI] (the slab layout of
 * moe_expert_ffn) -> dst device [n_experts][moe_q8_slab_bytes] (caller-owned).
 * moe_expert_ffn_q8: as moe_expert_ffn with a pool of quantised slabs (every
 * listed expert in a slot; no host pass); workspace of
 * moe_ffn_q8_workspace_bytes(T, H, k, I) bytes, 256-byte aligned; T*k <= 4096.
 * Errors: MOE_ERR_ARG on NULL pointers, H or I not a multiple of 16, too many
 * rows; MOE_ERR_ALIGN for unaligned pointers or a small workspace.
 */
size_t moe_q8_slab_bytes(int H, int I);
int moe_quantize_slabs(const void* src, int n_experts, int H, int I, void* dst, moe_stream_t stream);
size_t moe_ffn_q8_workspace_bytes(int T, int H, int k, int I);
int moe_expert_ffn_q8(const void* x, int T, int H, int I, int k, int E, const int32_t* offset, const int32_t* rows,
                      const int32_t* list_e, const int32_t* n_list, int max_list, const void* pool_q, int S,
                      const int32_t* e2s, float* y, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                      moe_stream_t stream);

/*
 * How GATHER mode serves a step that needs more experts than the pool holds
 * ("Porting vllm-expert-cache to NVIDIA GPUs", "Measuring, without fooling
 * yourself": a step is served from slots only when tokens x top_k <= slots;
 * count misses, not tokens).
 *   MOE_SCHED_CHUNKS  the step is cut into chunks of floor(S/k) consecutive
 *                     tokens, each managed, gathered, computed and combined in
 *                     turn (an expert needed by several chunks may be loaded
 *                     once per chunk).  Needs S >= k.
 *   MOE_SCHED_WAVES   each missing expert is loaded at most once per step.
 *                     Wave 0 is one manage call over the whole step: hits are
 *                     updated, and the misses (ascending id) take the slots
 *                     the step does not need while they last; the rest are
 *                     deferred.  The hits' FFN runs while wave 0's loads are
 *                     gathered on the side stream, then the loaded experts'
 *                     FFN.  Then the deferred experts follow in batches of at
 *                     most S (ascending id), each one manage call whose victims
 *                     may be any slot (its expert has been computed), a gather
 *                     and the batch's FFN.  One combine at the end.  An empty
 *                     batch changes nothing (stamp included).  Any S >= 1.
 * A step with T*k <= S, or S >= E, is one manage call under both.
 */
#define MOE_SCHED_CHUNKS 0
#define MOE_SCHED_WAVES 1

/* Arguments of moe_layer_forward.  Field meanings as in the calls above. */
typedef struct moe_layer_args {
  int32_t T, H, E, k, I, S;
  int32_t mode;   /* moe_mode */
  int32_t policy; /* moe_policy (GATHER: LRU or LFU; ZERO_RETURN: STATIC) */
  const void* x;             /* device bf16 [T][H] */
  const void* w_router;      /* device bf16 [H][E] */
  const float* logit_offset; /* device fp32 [E] or NULL */
  const float* sel_bias;     /* device fp32 [E] or NULL */
  void* pool;                /* device bf16 [S][3HI] slot pool */
  const void* host_slabs;    /* pinned host bf16 [E][3HI]; NULL in RESIDENT mode */
  int32_t* e2s;              /* device cache state (RESIDENT: e2s may be NULL = identity) */
  int32_t* s2e;
  uint32_t* prio;
  uint32_t* stamp;
  int32_t* ids;              /* device int32 [T][k] routing ids (output) */
  float* w;                  /* device fp32 [T][k] routing weights (output) */
  void* out;                 /* device bf16 [T][H] (output) */
  float* out_res;            /* device fp32 [T][H] (ZERO_RETURN output) */
  float* out_miss;           /* device fp32 [T][H] (ZERO_RETURN output) */
  int64_t* stats;            /* device int64 [4] or NULL: [0] += misses, [1] += manage calls, [2] += bytes gathered */
  int32_t* dev_status;       /* device int32 [1] */
  void* workspace;           /* device scratch, moe_layer_workspace_bytes() */
  size_t workspace_bytes;
  moe_prof* prof;            /* host struct, or NULL: per-kernel timing events */
  float affinity;            /* live-cache affinity lambda (0 = off); uses e2s before this step's manage */
  int32_t route_flags;       /* moe_route_ex flags (0 = softmax router, selection-only bias) */
  int32_t* window_counts;    /* device int32 [E] or NULL: each chunk's routings are added (moe_cache_count) */
  int32_t quant;             /* 0: bf16 slabs; 1: W8A8 slabs (moe_quantize_slabs), RESIDENT or GATHER mode */
  int32_t schedule;          /* GATHER steps larger than the pool: MOE_SCHED_CHUNKS or MOE_SCHED_WAVES */
  int32_t decode_kernels;    /* 0: persistent decode kernels where they apply (RESIDENT, GATHER); 1: separate */
} moe_layer_args;

/*
 * One MoE layer forward: route, then per chunk of tokens permute, manage,
 * gather on the side stream while the hit experts' FFN runs on the main
 * stream, the missed experts' FFN after the gather, and combine.
 * Sources: as for the calls above; "Betelgeuse: Running Qwen 3.8 Flash Next
 * ... on an RTX 3060", "What it actually does under the hood" (hits are
 * resolved on the device, no host sync inside the step, the decode pass
 * replays as one CUDA graph).
 * Steps larger than the pool (GATHER, S < E, T*k > S): token chunks or
 * expert waves, as args->schedule says (MOE_SCHED_*).  ZERO_RETURN (STATIC)
 * never chunks.
 * Small all-resident steps (RESIDENT, bf16, T <= 8, T*k <= 64, E <= 256,
 * H % 128 == 0 and H <= 2048, I % 128 == 0 and I <= 1024, no window counts,
 * decode_kernels == 0) run as one persistent cooperative launch, one CTA per
 * SM: router logits, a grid-wide wait, the top-k and grouping in every CTA,
 * the gate/up weight stream, the down weight stream (its weights loaded while
 * h is formed from the gate/up sums) and the combine.  W8A8 steps (quant = 1,
 * RESIDENT, T <= 8, T*k <= 64, E <= 256, H % 128 == 0 and H <= 2048,
 * I % 16 == 0 and I <= 1024, no window counts, decode_kernels == 0) have
 * their own persistent launch: router, the tokens' 8-bit codes, the gate/up
 * and down weight streams folded with dp4a (their exact int32 sums meet in
 * accumulators by integer atomics), h quantised per row, and the combine;
 * its output is bit for bit that of the separate W8A8 kernels.  Small
 * expert-cache steps (GATHER, LRU or LFU, T*k <= S <= 256, the shape limits
 * above, decode_kernels == 0, at least 96 SMs) run in the persistent
 * launches too, bf16 and W8A8 ("Porting vllm-expert-cache to NVIDIA GPUs",
 * "1. Kernels": a fused manager, gather and expert kernel): every CTA runs
 * the manage state machine on a shared-memory copy of the cache state, CTA 0
 * writes the new state, 48 CTAs copy the missing slabs from host memory into
 * their victim slots while the others stream the hit experts, and each
 * missing expert streams once its slab is in.  The state, miss count,
 * statistics and slot bytes are bit for bit those of the separate manage and
 * gather calls (and, with W8A8 slabs, the output too).  The grid-wide waits
 * of these kernels are bounded: a wait that gives up sets MOE_DEV_TIMEOUT
 * (an expert-cache step whose router wait gave up leaves the cache state,
 * statistics and pool as they were; a wait that gives up later, or in some
 * CTAs only, can leave the state and the pool disagreeing: reload both
 * before the next step).  They keep arrival counters at the start of the
 * workspace, which must therefore be zero-filled once before the first call
 * on it (each call leaves them zero).
 * `side` may be NULL or equal to `main` (then everything runs on `main`).
 * The sequence of launches depends only on the shapes, so it can be
 * captured into a CUDA graph.
 * Errors: as the calls above; MOE_ERR_CAPACITY if S < k in GATHER mode with
 * token chunks; MOE_ERR_ARG for an unknown schedule.
 */
int moe_layer_forward(const moe_layer_args* args, moe_stream_t main, moe_stream_t side);

/* Workspace of moe_layer_forward (device, 256-byte aligned, zero-filled once
 * before its first use: see above). */
size_t moe_layer_workspace_bytes(int T, int H, int E, int k, int I, int S);

/* The same size with the arguments in the order (T, H, I, E, k): the
 * workspace moe_layer_forward needs for up to T tokens in any mode, schedule
 * and pool size. */
size_t moe_workspace_bytes(int T, int H, int I, int E, int k);

#ifdef __cplusplus
}
#endif

#endif /* MOESLOT_H */
