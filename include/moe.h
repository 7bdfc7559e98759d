/*
 * moe.h — C ABI of the GB300 (sm_103a) offloading-aware MoE layer forward.
 *
 * One MoE layer forward in five stages, each a call below:
 *   1. moe_route            router softmax/top-k, APEX prefetch router,
 *                           ordinal-CDF budget delta_hat, top-(k+delta_hat)
 *                           prefetch set, delta* (metric)
 *   2. moe_select_resident  stall-free substitution / LoRE / fetch per miss
 *   3. moe_permute          token permutation by expert
 *      moe_expert_ffn       grouped SwiGLU expert FFN (+ shared experts)
 *   4. moe_lore             SPICE LoRE surrogate for LoRE slots
 *   5. moe_combine          gate-weighted combine plus shared experts
 * plus moe_stage_experts (pinned host -> HBM expert copies on a side stream)
 * and moe_layer_forward (all stages chained on one stream).
 * Beyond the single forward: moe_cache_update (a persistent expert cache
 * across decode steps), moe_prefetch_depth / moe_prefetch_min_depth (a
 * confidence-aware look-ahead over the next layers), moe_bitslice_pack /
 * moe_bitslice_ffn (a low-precision draft FFN on bit-sliced INT8 weights) and
 * the heterogeneous CPU-GPU path: moe_hetero_fetch_min_rows,
 * moe_select_hetero, moe_cpu_experts and moe_layer_forward_hetero (exact
 * host execution of high-confidence misses chosen by a cost model).
 *
 * Conventions (all entry points):
 *   - Every function returns moe_status (the two size helpers and
 *     moe_prefetch_min_depth return their value); nothing aborts, traps,
 *     throws or prints.  Host-detectable argument errors are returned before any work
 *     is queued.  Errors found by a kernel (a bad expert index, an available
 *     set smaller than k, a timed-out wait) are recorded in the device error
 *     word inside the workspace and reported by moe_check().
 *   - Pointers are DEVICE pointers unless the name starts with host_.
 *     The caller allocates and owns every buffer, including the workspace
 *     (size from moe_workspace_size) and the expert table (size from
 *     moe_expert_table_size).  The library allocates no memory.
 *   - All work is queued asynchronously on the caller's stream
 *     (a cudaStream_t passed as void*; NULL = the legacy default stream).
 *     Only moe_check(), moe_expert_table_init() and moe_stage_experts()'s
 *     host-side bookkeeping synchronise.
 *   - Row-major layouts throughout.  Activations and weights share the
 *     layer's weight type (MOE_DTYPE_BF16 or MOE_DTYPE_F32); router
 *     probabilities, gates and outputs are float32; indices int32; expert
 *     sets are uint64 bitmasks (bit e = expert e, so N <= 64).
 *   - Ties are broken towards the lowest expert / channel index.
 *
 * Sources (page titles and sections):
 *   APEX: Adaptive Expert Prefetching for Edge MoE Inference (blog write-up),
 *     §4.1 prefetch router, §4.2 delta* and the ordinal-logistic CDF,
 *     §4.3 execution modes and Algorithm 1 (stall_free_select).
 *   SPICE: Speculative Prefetching with Low-Rank Expert Surrogates and
 *     Heterogeneous Orchestration for MoE Inference (PaperDaily write-up),
 *     sections on the LoRE low-rank surrogate, CPU-GPU orchestration and
 *     confidence-aware adaptive prefetch.
 *   ELMoE-3D (CSDN post): expert-axis elasticity (heat statistics, top-K
 *     subset, heat decay) and the bit-slicing section with its data-layout
 *     note.
 *   FloE: On-the-Fly MoE Inference on Memory-constrained GPU (paper notes),
 *     method §1 (contextual sparsity forward), §3 (sparse GEMV, compact
 *     asynchronous transfer).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* NULL where a buffer is required, bad size, misaligned pointer */
    MOE_ERR_UNSUPPORTED = 2,   /* N > 64, k > 8, d not a multiple of 256, dtype not handled */
    MOE_ERR_CAPACITY = 3,      /* workspace/table too small, or (device) |A_t| < k */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch, copy, event) */
    MOE_ERR_STAGING = 5,       /* an expert copy could not be queued */
    MOE_ERR_TIMEOUT = 6,       /* (device) a bounded wait inside a kernel gave up */
    MOE_ERR_DEVICE_INDEX = 7   /* (device) an expert or slot index out of range */
} moe_status;

typedef enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 } moe_dtype;

/* What happens to a routed expert that is not in the available set A_t. */
typedef enum {
    MOE_MISS_EXACT = 0,       /* fetch it and compute it: output = plain MoE (APEX §4.3,
                                 correctness-preserving mode) */
    MOE_MISS_SUBSTITUTE = 1,  /* stall-free substitution (APEX §4.3, Algorithm 1) */
    MOE_MISS_LORE = 2,        /* LoRE surrogate y_shared + B_e A_e x (SPICE, LoRE section) */
    MOE_MISS_HYBRID = 3,      /* router prob < gamma -> LoRE, else substitute */
    MOE_MISS_HETERO = 4       /* router prob < gamma -> LoRE, else exact: fetched to the GPU
                                 or computed on the host, per expert by the cost model
                                 (SPICE, CPU-GPU collaboration); moe_select_hetero only */
} moe_miss_policy;

/* Kind of each final slot.  CPU: an exact expert computed on the host cores
 * (moe_cpu_experts) and merged in the combine like a computed slot. */
typedef enum {
    MOE_KIND_COMPUTE = 0, MOE_KIND_FETCH = 1, MOE_KIND_LORE = 2, MOE_KIND_CPU = 3
} moe_slot_kind;

/* Layer dimensions.  T: tokens in this call (<= the T the workspace was sized
 * for); d: hidden size (multiple of 256); N: routed experts (<= 64);
 * k: top-k (<= 8); I: routed-expert intermediate size (multiple of 64);
 * n_shared / I_shared: shared experts and their intermediate size;
 * r: LoRE rank (0: no LoRE factors); delta_max: largest prefetch budget
 * (N - k); wtype: weight/activation type; renorm_topk: 1 to renormalise the
 * final gates over the final set (0: gates are the router probabilities). */
typedef struct {
    int T, d, N, k, I, n_shared, I_shared, r, delta_max;
    moe_dtype wtype;
    int renorm_topk;
} moe_dims;

/* Slot counters written by moe_select_resident (int32[MOE_NUM_COUNTERS]). */
enum {
    MOE_CNT_HIT = 0,        /* routed and available: computed as routed */
    MOE_CNT_SUBSTITUTE = 1, /* slots given to a substitute expert */
    MOE_CNT_LORE = 2,       /* slots served by the LoRE surrogate */
    MOE_CNT_FETCH = 3,      /* slots whose expert must be fetched (EXACT) */
    MOE_CNT_OVERLAP = 4,    /* tokens whose routed set lies inside their prefetch set */
    MOE_CNT_DELTA_HAT = 5,  /* sum over tokens of delta_hat */
    MOE_CNT_DELTA_STAR = 6, /* sum over tokens of delta* */
    MOE_CNT_SHORTFALL = 7,  /* tokens whose available set had fewer than k experts */
    MOE_CNT_CPU = 8,        /* slots computed on the host cores (HETERO) */
    MOE_NUM_COUNTERS = 9
};

const char* moe_status_string(moe_status s);

/* Bytes of device workspace needed for calls with these dims (T = the
 * largest token count that will be passed).  The workspace holds router
 * logits, the permutation plan, FFN intermediates and partial sums, and the
 * device error word.  Zero-fill it once before first use (its error word
 * must start clear); moe_check() clears the error word after reading it. */
moe_status moe_workspace_size(const moe_dims* dims, size_t* bytes);

/* Bytes of device memory for the expert table (per-expert weight pointers
 * and TMA descriptors for N routed + n_shared shared experts). */
moe_status moe_expert_table_size(const moe_dims* dims, size_t* bytes);

/* Fill the expert table from HOST arrays of DEVICE pointers.
 * host_w_gate/up/down[e]: expert e's [I, d] matrices (row i = intermediate
 * channel i for all three: up/gate rows are the input projections of channel
 * i, down row i is channel i's output projection).  host_sh_gate/up/down[s]:
 * shared expert s's [I_shared, d] matrices (may be NULL if n_shared == 0).
 * Every matrix must be 16-byte aligned.  Entries may point into one [N, I, d]
 * block or anywhere else (a slot of an expert cache).  Synchronises `stream`.
 * Call again after an expert moves to a new address. */
moe_status moe_expert_table_init(const moe_dims* dims,
                                 const void* const* host_w_gate, const void* const* host_w_up,
                                 const void* const* host_w_down,
                                 const void* const* host_sh_gate, const void* const* host_sh_up,
                                 const void* const* host_sh_down,
                                 void* table, size_t table_bytes, void* stream);

/* Stage 1 — router and prefetch router (APEX §4.1-§4.2).
 *   x [T,d]: layer input.  w_router [N,d], router_bias [N] (float32, NULL = none):
 *   router logits l = x w_router^T + b; router_prob [T,N] = softmax(l);
 *   topk_idx [T,k] = the k largest logits (descending, lowest index first on
 *   ties); topk_gate [T,k] = router_prob of those experts.
 *   x_pre [T,d] (NULL = x): input of the prefetch router (pre-attention state);
 *   w_prefetch [N,d] (NULL = no prefetch router: delta_hat = 0, prefetch_mask
 *   = all ones, delta_star = 0); w_ord [d] float32 and theta [delta_max+1]
 *   float32 (non-decreasing): the ordinal-logistic CDF
 *   p_delta = sigmoid(theta_delta - w.x_pre); delta_hat [T] = min{delta :
 *   p_delta >= tau}, delta_max if none; prefetch_mask [T] = top-(k+delta_hat)
 *   of the prefetch logits; delta_star [T] (NULL = skip) = min{delta : routed
 *   set within top-(k+delta)}.
 *   n_resident > 0 with batch_resident (device uint64, 1 element) also writes
 *   the n_resident experts with the largest prefetch probability summed over
 *   the T tokens (the set a prefetcher would stage for this batch).
 * Errors: INVALID_ARG (NULL required buffer, tau outside (0,1)),
 * UNSUPPORTED, CAPACITY (workspace too small), CUDA. */
moe_status moe_route(const moe_dims* dims, const void* x, const void* w_router,
                     const float* router_bias, const void* x_pre, const void* w_prefetch,
                     const float* w_ord, const float* theta, float tau, int n_resident,
                     int32_t* topk_idx, float* topk_gate, float* router_prob,
                     int32_t* delta_hat, uint64_t* prefetch_mask, int32_t* delta_star,
                     uint64_t* batch_resident, void* ws, size_t ws_bytes, void* stream);

/* Stage 2 — miss handling (APEX §4.3 and Algorithm 1; SPICE LoRE section).
 *   Available set A_t = resident (device uint64, NULL = all experts) AND
 *   prefetch_mask[t] (NULL = all experts).  A routed expert outside A_t is
 *   handled by `policy` (moe_miss_policy); HYBRID sends it to LoRE when its
 *   router probability is below gamma and to substitution otherwise.
 *   Substitutes are the available, non-routed experts with the largest
 *   ORIGINAL router probability; each substitute carries its own probability
 *   as gate.  Outputs, k slots per token in descending router probability:
 *   final_idx [T,k], final_gate [T,k] (renormalised if dims->renorm_topk),
 *   final_kind [T,k] (moe_slot_kind); fetch_mask (device uint64, NULL = skip)
 *   = OR of the experts with a FETCH slot; counters (device int32
 *   [MOE_NUM_COUNTERS], NULL = skip).  delta_hat, delta_star (NULL = skip)
 *   only feed the counters.
 *   A token whose A_t has fewer than k experts under SUBSTITUTE or HYBRID
 *   keeps what it can, counts in MOE_CNT_SHORTFALL and sets MOE_ERR_CAPACITY
 *   in the device error word.  LORE and HYBRID need dims->r > 0 (else
 *   INVALID_ARG). */
moe_status moe_select_resident(const moe_dims* dims, const float* router_prob,
                               const int32_t* topk_idx, const uint64_t* prefetch_mask,
                               const uint64_t* resident, int policy, float gamma,
                               const int32_t* delta_hat, const int32_t* delta_star,
                               int32_t* final_idx, float* final_gate, int32_t* final_kind,
                               uint64_t* fetch_mask, int32_t* counters,
                               void* ws, size_t ws_bytes, void* stream);

/* Pinned host -> HBM copies of the experts in host_fetch_mask (a HOST value:
 * read the device fetch_mask first), for the EXACT policy.  For each expert
 * e in the mask, copies host_w_{gate,up,down}[e] (pinned host, [I,d] each)
 * to dev_w_{gate,up,down}[e] (device) with cudaMemcpyAsync on stage_stream,
 * then records done_event (a cudaEvent_t as void*) on stage_stream; the
 * compute stream waits on that event before moe_expert_ffn.  *bytes receives
 * the bytes queued.  Errors: INVALID_ARG, STAGING (a copy or the event
 * record could not be queued; nothing further is queued). */
moe_status moe_stage_experts(const moe_dims* dims, uint64_t host_fetch_mask,
                             const void* const* host_w_gate, const void* const* host_w_up,
                             const void* const* host_w_down,
                             void* const* dev_w_gate, void* const* dev_w_up,
                             void* const* dev_w_down, void* stage_stream, void* done_event,
                             size_t* bytes);

/* Heterogeneous CPU-GPU orchestration (SPICE write-up, section on CPU-GPU
 * collaboration for prefetch misses, Fig. 6 and its cost model).  A routed
 * expert outside the available set whose router probability is at least
 * gamma must be computed exactly; it is either fetched (its weights copied
 * to the GPU, then computed there) or computed on the host cores from the
 * host copy of its weights, with only the token rows crossing the link.  Per
 * missing expert e with n_e such token rows in the batch:
 *   fetch cost = W_e / B + T_gpu          CPU cost = n_e * (t_cpu + 2 H / B)
 * and e is fetched iff the fetch cost is the smaller (ties go to the host).
 * Times in seconds, sizes in bytes. */
typedef struct {
    double link_bytes_per_s;  /* B: host <-> device link bandwidth */
    double expert_bytes;      /* W_e: one routed expert's gate, up and down matrices */
    double gpu_expert_s;      /* T_gpu: one routed expert's FFN on the GPU */
    double cpu_row_s;         /* t_cpu: one token row of one expert's FFN on the host */
    double hidden_bytes;      /* H: one token's hidden state (d x element size) */
} moe_hetero_cost;

/* The smallest n_e for which fetching wins under *cost (1 if it always
 * wins; INT32_MAX if it never does).  Host only; -1 for a negative, NaN or
 * missing parameter or a non-positive bandwidth. */
int moe_hetero_fetch_min_rows(const moe_hetero_cost* cost);

/* Miss handling of the heterogeneous path: moe_select_resident with
 * MOE_MISS_HETERO (router prob < gamma -> LoRE, needs dims->r > 0 when
 * gamma > 0), then per missing expert: n_e >= fetch_min_rows -> its slots
 * are FETCH, else CPU.  Also places the CPU slots after the GPU segments of
 * the permutation: with n_gpu the number of COMPUTE and FETCH slots, the j-th
 * CPU slot (t, s) in slot order gets inv_perm[t*k+s] = n_gpu + j and
 * perm[n_gpu + j] = t*k+s; moe_permute, called next, fills the entries of
 * the other slots and leaves these.  fetch_mask / cpu_mask (device uint64,
 * may be NULL) = the experts with FETCH / CPU slots; counters as in
 * moe_select_resident plus MOE_CNT_CPU (MOE_CNT_FETCH counts only the slots
 * left to fetch).  Errors as moe_select_resident; INVALID_ARG also for
 * fetch_min_rows < 1. */
moe_status moe_select_hetero(const moe_dims* dims, const float* router_prob, const int32_t* topk_idx,
                             const uint64_t* prefetch_mask, const uint64_t* resident, float gamma,
                             int fetch_min_rows, const int32_t* delta_hat, const int32_t* delta_star,
                             int32_t* final_idx, float* final_gate, int32_t* final_kind, int32_t* perm,
                             int32_t* inv_perm, uint64_t* fetch_mask, uint64_t* cpu_mask, int32_t* counters,
                             void* ws, size_t ws_bytes, void* stream);

/* Host scratch bytes moe_cpu_experts needs for dims (T*k*I*4 plus
 * bookkeeping; 0 for bad dims). */
size_t moe_cpu_experts_scratch_size(const moe_dims* dims);

/* The host side of the heterogeneous path: every CPU slot's expert FFN,
 * computed exactly on the host cores from the host copy of the weights
 * (bf16 or float32 values, float32 arithmetic):
 *   y_rows[j] = (SiLU(x_t Wg_e^T) (.) x_t Wu_e^T) Wd_e   (ungated)
 * for the j-th CPU slot (t, s) in slot order, e = final_idx[t*k+s].
 * HOST pointers, all of them: host_x [T, d] (layer type), host_final_idx /
 * host_final_kind [T, k] (copies of moe_select_hetero's outputs),
 * host_w_gate/up/down[e] ([I, d] each), host_y_rows [T*k, d] float32,
 * scratch of moe_cpu_experts_scratch_size bytes.  n_threads <= 0: every core
 * of the process's affinity mask.  *n_rows = the CPU slots computed;
 * *first_row = n_gpu, the y_perm row of the first of them (copy the rows
 * there before moe_combine).  The work of one call is spread over a pool of
 * host threads that the library starts on first use and keeps.  The result
 * does not depend on n_threads.  No CUDA call.  Errors: INVALID_ARG (NULL,
 * an index out of range, scratch too small), UNSUPPORTED (dims). */
moe_status moe_cpu_experts(const moe_dims* dims, const void* host_x, const int32_t* host_final_idx,
                           const int32_t* host_final_kind, const void* const* host_w_gate,
                           const void* const* host_w_up, const void* const* host_w_down, int n_threads,
                           float* host_y_rows, void* scratch, size_t scratch_bytes, int32_t* n_rows,
                           int32_t* first_row);

/* Stage 3a — token permutation by expert.
 *   Slots (t, s) of kind COMPUTE or FETCH are grouped by expert, stable in
 *   (t, s) order.  expert_offsets [N+1]: exclusive scan of per-expert counts;
 *   perm [T*k]: perm[pos] = t*k + s for pos < expert_offsets[N];
 *   inv_perm [T*k]: position of slot (t, s), -1 for LoRE slots.
 *   Also writes the FFN work plan into the workspace. */
moe_status moe_permute(const moe_dims* dims, const int32_t* final_idx,
                       const int32_t* final_kind, int32_t* expert_offsets, int32_t* perm,
                       int32_t* inv_perm, void* ws, size_t ws_bytes, void* stream);

/* Stage 3b — grouped SwiGLU FFN over the permuted slots and the shared
 * experts: y = (SiLU(X W_gate^T) (.) X W_up^T) W_down per expert (FloE method
 * §1 with S_t = identity when keep_frac == 1).
 *   x [T,d]; table: from moe_expert_table_init; expert_offsets/perm from
 *   moe_permute (same call sequence, same workspace).
 *   keep_frac in (0,1]: < 1 applies FloE contextual sparsity to routed
 *   experts (keep the m = ceil(keep_frac*I) channels with the largest
 *   |x.W_up| per token, lowest channel index among equal values; gate and
 *   down rows read only for the union of the kept channels of an expert's
 *   tokens, each token using its own mask).  Decode batches (T <= 64) of
 *   bf16 layers only; otherwise MOE_ERR_UNSUPPORTED.
 *   y_perm [T*k, d] float32: row pos = the expert output for slot perm[pos]
 *   (ungated); y_shared [T, d] float32 (NULL if n_shared == 0) = sum of the
 *   shared experts' outputs.  x must be 16-byte aligned, and so must y_perm
 *   and y_shared for batches of more than 64 tokens (MOE_ERR_INVALID_ARG
 *   otherwise).
 *   Kernels (moe_expert_ffn_path names the choice for a call): batches of
 *   more than 64 tokens of bf16 layers run as a tcgen05 tensor-core grouped
 *   GEMM; dense bf16 batches of 4..64 tokens (d a multiple of 128, expert
 *   widths multiples of 16) as a tcgen05 GEMM with the weight rows on the
 *   MMA's M side; the rest (1..3 tokens, fp32 layers, FloE) as an
 *   HBM-streaming CUDA-core GEMV (for one token of a dense bf16 layer with
 *   d = 1536 or 2048, one channel per warp). */
moe_status moe_expert_ffn(const moe_dims* dims, const void* x, const void* table,
                          const int32_t* expert_offsets, const int32_t* perm, float keep_frac,
                          float* y_perm, float* y_shared, void* ws, size_t ws_bytes,
                          void* stream);

/* Which kernels moe_expert_ffn runs for these dimensions and keep_frac: a
 * static string, "tc-prefill" (gather + two tensor-core GEMM launches),
 * "tc-decode" (tensor-core GEMM + partial-row reduction, and a row gather
 * first for batches of 17..64 tokens), "gemv" (CUDA-core GEMV + reduction),
 * "gemv-1tok" (the one-token CUDA-core GEMV, a channel per warp, +
 * reduction), "gemv-floe" (FloE preparation + sparse GEMV + reduction) or
 * "unsupported".  No device work. */
const char* moe_expert_ffn_path(const moe_dims* dims, float keep_frac);

/* Diagnostic: where the last moe_expert_ffn call with keep_frac < 1 left the
 * FloE kept-channel bitsets inside `ws` (FloE method §1, the mask S_t):
 * *kept = device uint32 [rows][*words_per_row], one row per permuted
 * position (the order of perm), bit i = channel i kept.  Valid until the
 * next call that uses the workspace. */
moe_status moe_floe_kept_mask(const moe_dims* dims, void* ws, size_t ws_bytes, const uint32_t** kept,
                              int32_t* words_per_row);

/* moe_expert_ffn without a workspace, for callers that cannot allocate device
 * memory when they run the layer: an engine plugin handed only its inputs and
 * outputs (the host engine owns the whole memory budget), or a decode loop
 * that cannot pay the device-wide synchronisation of cudaMalloc/cudaFree.
 * The source pages have no counterpart of this call; it is a deployment
 * convenience.
 *   Same inputs and outputs as moe_expert_ffn (dense experts only, i.e.
 *   keep_frac = 1), with expert_offsets/perm from moe_permute.  The plan,
 *   partial sums and error word live in a 16 MiB array that the library
 *   holds on every GPU it is loaded on, until the process exits.  Batches
 *   whose scratch would exceed 16 MiB are rejected with MOE_ERR_CAPACITY
 *   before anything is queued (decode sizes fit: e.g. 32 tokens at d = 2048
 *   or d = 4096).  device_status (device int32[2], may be NULL) receives the
 *   call's device error code and detail when its kernels have run.
 *   The first call in a CUDA context looks the array's address up
 *   (cudaGetSymbolAddress) and remembers it under the context's unique ID,
 *   so a context made after cudaDeviceReset, or a non-primary one, gets its
 *   own lookup; make that first call outside of any stream capture.
 *   All calls share the array: calls
 *   whose kernels overlap on the GPU race, so order them on one stream.
 *   Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call. */
moe_status moe_expert_ffn_noalloc(const moe_dims* dims, const void* x, const void* table,
                                  const int32_t* expert_offsets, const int32_t* perm,
                                  float* y_perm, float* y_shared, int32_t* device_status,
                                  void* stream);

/* Stage 4 — LoRE surrogate residual (SPICE, LoRE section):
 *   y_lore[t] = sum over LoRE slots s of final_gate[t,s] * B_e (A_e x_t),
 *   e = final_idx[t,s]; zero rows for tokens without LoRE slots.
 *   lore_a [N, r, d], lore_b [N, d, r] in the layer's weight type;
 *   y_lore [T, d] float32 (written).  The rank-r projections A_e x_t go
 *   through the workspace. */
moe_status moe_lore(const moe_dims* dims, const void* x, const int32_t* final_idx,
                    const int32_t* final_kind, const float* final_gate, const void* lore_a,
                    const void* lore_b, float* y_lore, void* ws, size_t ws_bytes, void* stream);

/* Look-ahead layers handled by one moe_prefetch_depth call, at most. */
#define MOE_MAX_AHEAD 16

/* Confidence-aware prefetch depth (beyond the single layer forward; SPICE
 * write-up, section on confidence-aware adaptive prefetch).  A draft predicts
 * the expert distribution of each of the next n_ahead layers from the current
 * hidden state x; the draft head is the identity here (look-ahead layer j's
 * router applied to x).  For every token t and look-ahead layer j:
 *   logits_ahead[j][t][e] = x_t . w_router_ahead[j][e] (+ bias_ahead[j][e])
 *   conf[t][j]  = the probability mass (softmax over the N logits) on the
 *                 top-k experts (k = dims->k; largest logits, lower index on
 *                 ties)
 *   depth[t]    = min(n_ahead, max(d_min, c)), c = the number of leading
 *                 layers j = 0, 1, ... with conf >= tau (the scan stops at the
 *                 first layer below tau)
 *   token_masks[t][j] = the top-k set of layer j if j < depth[t], else 0
 *   layer_masks[j]    = OR over tokens of token_masks[t][j]: the experts to
 *                 stage for look-ahead layer j.
 * x [T, d] and each w_router_ahead[j] [N, d] in the layer's weight type,
 * 16-byte aligned; bias_ahead NULL or an array of n_ahead device pointers
 * ([N] float32, entries may be NULL); w_router_ahead and bias_ahead are HOST
 * arrays of device pointers.  logits_ahead [n_ahead, T, N] float32, conf
 * [T, n_ahead] float32, depth [T] int32, token_masks [T, n_ahead] and
 * layer_masks [n_ahead] uint64: device, written.  d_min comes from
 * moe_prefetch_min_depth.  Errors: INVALID_ARG (n_ahead outside
 * 1..MOE_MAX_AHEAD, d_min < 0, tau not finite, a NULL or misaligned buffer),
 * UNSUPPORTED (N > 64).  Asynchronous. */
moe_status moe_prefetch_depth(const moe_dims* dims, int n_ahead, const void* x,
                              const void* const* w_router_ahead, const float* const* bias_ahead, float tau,
                              int d_min, float* logits_ahead, float* conf, int32_t* depth,
                              uint64_t* token_masks, uint64_t* layer_masks, void* ws, size_t ws_bytes,
                              void* stream);

/* The minimum prefetch depth (SPICE write-up, same section):
 * ceil(expert_bytes / (link_bytes_per_s * layer_seconds)), the layers a
 * transfer of one expert must start ahead so that it lands before its layer
 * runs.  A quotient within 1e-9 (relative) of an integer counts as that
 * integer.  Host only, no device work; -1 for a negative size, a
 * non-positive bandwidth or layer time, or a depth above INT32_MAX. */
int moe_prefetch_min_depth(double expert_bytes, double link_bytes_per_s, double layer_seconds);

/* Bit-sliced expert weights (beyond the single layer forward; ELMoE-3D,
 * bit-slicing section and its data-layout note): a low-precision draft of the
 * expert FFN.  Each weight is an INT8 value q with a scale per output row
 * (s_r = max |W[r][.]| / 127, q = rint(W / s_r) clamped to +-127, float32
 * arithmetic); its 8 bits are stored as binary planes and a b-bit weight is
 * s_r times the top b planes recombined (plane 7 carries -128, plane p < 7
 * carries 2^p: the value floored to a multiple of 2^(8-b)).
 *
 * moe_bitslice_pack: W [rows, cols] row-major in wtype (device); transpose
 * != 0 packs W^T.  With (R, C) = (rows, cols), or (cols, rows) transposed,
 * C a multiple of 32: planes [8][R][C/32] uint32, slot s = plane 7 - s (the
 * top b planes are the first b*R*C/32 words), bit i of word w of row r =
 * that plane's bit of q[r][32w + i]; scales [R] float32.  Device, written.
 * Errors: INVALID_ARG (sizes, C not a multiple of 32, NULL), UNSUPPORTED
 * (wtype).  Asynchronous. */
moe_status moe_bitslice_pack(int rows, int cols, moe_dtype wtype, const void* w, int transpose,
                             uint32_t* planes, float* scales, void* stream);

/* Scratch bytes moe_bitslice_ffn needs for T tokens of `slots` slots each
 * (k + n_shared): T*slots*(I + d)*4 + T*(d/16)*4 (0 for bad sizes). */
size_t moe_bitslice_scratch_size(int d, int I, int T, int slots);

/* The draft FFN with b-bit weights for T tokens of k routed slots and the
 * n_shared shared experts:
 *   y[t] (+)= sum over routed slots s, in order, of gate[t][s] *
 *             FFN_b(idx[t][s], x_t), then + FFN_b(N + i, x_t) for every
 *             shared expert i, in order
 *   FFN_b(e, x) = Wd_b^T-rows . (SiLU(Wg_b x) (.) Wu_b x)   (float32 math)
 * planes_gate / planes_up: the N routed and then the n_shared shared
 * experts' [I, d] gate / up matrices packed one after another
 * ([N + n_shared][8][I][d/32], scales [N + n_shared][I]); planes_down: their
 * W_down [I, d] packed transposed ([N + n_shared][8][d][I/32], scales
 * [N + n_shared][d]); x [T, d] in xtype; idx [T, k] int32 (a routed slot
 * naming no expert in 0..N-1 contributes 0); gate [T, k] float32 or NULL
 * (every gate 1); accumulate != 0 adds to y [T, d] float32, else overwrites
 * it; scratch of moe_bitslice_scratch_size(d, I, T, k + n_shared) bytes.
 * All device pointers, planes and x 16-byte aligned.  d and I multiples of
 * 32, d <= 4096, I <= 4096, T * (k + n_shared) <= 65535, bits in 1..8.  Errors: INVALID_ARG, UNSUPPORTED
 * (xtype, sizes beyond those).  Asynchronous. */
moe_status moe_bitslice_ffn(int d, int I, int N, int n_shared, int bits, moe_dtype xtype, const void* x, int T, int k,
                            const int32_t* idx, const float* gate, const uint32_t* planes_gate,
                            const float* scales_gate, const uint32_t* planes_up, const float* scales_up,
                            const uint32_t* planes_down, const float* scales_down, int accumulate, float* y,
                            void* scratch, size_t scratch_bytes, void* stream);

/* Persistent expert cache across decode steps (beyond the single layer
 * forward; ELMoE-3D, expert-axis elasticity: heat statistics of the experts
 * the routing function selects, the most frequently activated top-K kept
 * resident and refreshed as the pattern drifts, heat decaying by a factor
 * just below 1 each step).  One step, after the layer ran with its resident
 * mask = *cache_mask (moe_layer_args.resident, n_resident = 0):
 *   heat[e]     <- decay * heat[e] + #{slots of topk_idx routed to e}
 *                  (float32, a rounded product then a rounded sum)
 *   *cache_mask <- the `capacity` experts of largest heat, lowest index on
 *                  ties (every expert if capacity >= N)
 *   *admit_mask <- new cache & ~old cache: the experts to stage in before the
 *                  next step (may be NULL)
 *   stats[0..3] += routed slots whose expert was in the old cache (hits),
 *                  routed slots, experts admitted, experts evicted (stats may
 *                  be NULL; the caller zeroes it).
 * topk_idx [T, k] int32 (moe_route's routed experts, before miss handling);
 * heat [N] float32, cache_mask / admit_mask uint64, stats int32[4]: device
 * pointers.  Errors: INVALID_ARG (NULL topk_idx / heat / cache_mask, decay
 * outside [0, 1], capacity < 0), UNSUPPORTED (N > 64).  Asynchronous. */
moe_status moe_cache_update(const moe_dims* dims, const int32_t* topk_idx, float decay, int capacity,
                            float* heat, uint64_t* cache_mask, uint64_t* admit_mask, int32_t* stats,
                            void* stream);

/* Stage 5 — combine:
 *   out[t] = y_shared[t] * (1 + sum of LoRE-slot gates)
 *          + sum over COMPUTE/FETCH slots of final_gate * y_perm[inv_perm[t,s]]
 *          + y_lore[t]
 *   (the LoRE slot stands for y_shared + B_e A_e x, SPICE LoRE section).
 *   Slots are summed in slot order (deterministic).  y_shared, y_lore may be
 *   NULL (zero).  out [T, d] float32. */
moe_status moe_combine(const moe_dims* dims, const float* y_perm, const int32_t* inv_perm,
                       const float* final_gate, const int32_t* final_kind,
                       const float* y_shared, const float* y_lore, float* out, void* stream);

/* All stages for one layer on one stream (no host synchronisation).  FETCH
 * slots are computed from the table's current pointers: stage them first
 * (moe_stage_experts) when the policy is EXACT. */
typedef struct {
    const void* x; const void* x_pre;
    const void* w_router; const float* router_bias;
    const void* w_prefetch; const float* w_ord; const float* theta; float tau;
    int n_resident;               /* > 0: batch resident set from the prefetch router */
    const uint64_t* resident;     /* used when n_resident <= 0 (NULL = all) */
    int use_prefetch_mask;        /* A_t includes the per-token prefetch set */
    int policy; float gamma; float keep_frac;
    const void* table; const void* lore_a; const void* lore_b;
} moe_layer_args;

typedef struct {
    int32_t* topk_idx; float* topk_gate; float* router_prob; int32_t* delta_hat;
    uint64_t* prefetch_mask; int32_t* delta_star; uint64_t* batch_resident;
    int32_t* final_idx; float* final_gate; int32_t* final_kind; uint64_t* fetch_mask;
    int32_t* counters; int32_t* expert_offsets; int32_t* perm; int32_t* inv_perm;
    float* y_perm; float* y_shared; float* y_lore; float* out;
} moe_layer_outputs;

moe_status moe_layer_forward(const moe_dims* dims, const moe_layer_args* args,
                             const moe_layer_outputs* outs, void* ws, size_t ws_bytes,
                             void* stream);

/* moe_layer_forward with the input and the output in host memory: copies
 * host_x ([T, d], the layer's type) into args->x, runs the layer, copies
 * outs->out ([T, d] float32) to host_out, all queued on `stream` (pinned host
 * buffers make the copies asynchronous; synchronise before reading
 * host_out).  Replayed as one CUDA graph per argument set, like
 * moe_layer_forward, the copies included.  args->x_pre must be NULL or x.
 * Errors: those of moe_layer_forward, INVALID_ARG for missing buffers. */
moe_status moe_layer_forward_host(const moe_dims* dims, const moe_layer_args* args,
                                  const moe_layer_outputs* outs, const void* host_x, float* host_out,
                                  void* ws, size_t ws_bytes, void* stream);

/* moe_layer_forward replays CUDA graphs: the first call with a given set of
 * arguments (the bytes of dims, args and outs, the workspace and the device)
 * on a non-default stream that is not being captured captures the call's
 * launch sequence into a graph; later calls with the same arguments launch
 * that graph (one host call instead of one per kernel).  The buffers are
 * read at replay time, so their contents may change between calls; a call
 * made while the caller captures its own graph, or on the legacy default
 * stream, launches the kernels directly.  Up to 48 graphs are kept (least
 * recently used replaced).  enabled = 0 turns replay off for later calls. */
void moe_set_graph_replay(int enabled);

/* Host buffers of moe_layer_forward_hetero (pinned host memory, caller-owned;
 * sized for dims->T). */
typedef struct {
    void* x;              /* [T, d] layer type: the hidden state staged to the host */
    int32_t* final_idx;   /* [T, k] */
    int32_t* final_kind;  /* [T, k] */
    uint64_t* masks;      /* [2]: fetch mask, CPU mask */
    float* y_rows;        /* [T*k, d] float32: CPU-slot outputs */
    void* scratch;        /* moe_cpu_experts scratch */
    size_t scratch_bytes;
} moe_hetero_host;

/* What one moe_layer_forward_hetero call did. */
typedef struct {
    int32_t cpu_slots;        /* slots computed on the host */
    int32_t fetch_experts;    /* experts copied to the GPU */
    int32_t fetch_min_rows;   /* the cost model's threshold */
    int32_t lore_slots;       /* slots served by LoRE */
    double fetch_bytes;       /* expert bytes queued host -> device */
    double cpu_link_bytes;    /* token rows down and CPU results up */
    double host_ms;           /* host FFN time */
    double wait_ms;           /* time the host waited for the routing decisions */
} moe_hetero_stats;

/* One layer forward on the heterogeneous path, orchestrated in three steps
 * (SPICE, Fig. 6): (1) routing and miss handling run on `stream`, then the
 * hidden state and the decisions are copied to host->* and the host waits
 * for them; (2) the fetched experts' copies are queued on stage_stream
 * (moe_stage_experts into dev_w_*, stage_event recorded, `stream` waits on
 * it), the GPU experts, LoRE and the shared experts are queued on `stream`,
 * and meanwhile the host cores compute the CPU slots (moe_cpu_experts);
 * (3) the CPU rows are copied into y_perm and moe_combine merges every slot.
 * args->policy is ignored (HETERO with args->gamma); args->keep_frac must be
 * 1 and args->x_pre NULL or x.  Returns when step 3 is queued; host->y_rows
 * must stay untouched until `stream` has passed it.  *stats (may be NULL).
 * Errors: those of the stages, CUDA, STAGING. */
moe_status moe_layer_forward_hetero(const moe_dims* dims, const moe_layer_args* args,
                                    const moe_layer_outputs* outs, const moe_hetero_cost* cost,
                                    const void* const* host_w_gate, const void* const* host_w_up,
                                    const void* const* host_w_down, void* const* dev_w_gate,
                                    void* const* dev_w_up, void* const* dev_w_down,
                                    const moe_hetero_host* host, int n_threads, void* ws, size_t ws_bytes,
                                    void* stream, void* stage_stream, void* stage_event,
                                    moe_hetero_stats* stats);

/* Overlapped expert-cache pipeline for decode loops (beyond the single
 * layer forward; ELMoE-3D expert-axis elasticity with its heat decay; SPICE
 * write-up, confidence-aware prefetch: copies must start D_min =
 * ceil(W_e / (B T_layer)) layers ahead to land in time).  The layer runs on
 * resident = cache & landed, where `landed` holds the experts whose weights
 * have arrived.  Each step queues, with no host synchronisation on the step
 * path: the layer forward; the heat / cache update (moe_cache_update's
 * rule), which also forms the next step's resident set from the host's
 * landed mask (passed by value); and a read-back of the masks (written by
 * that kernel straight into the pinned ring when the ring is mapped into
 * the device's address space, else copied).  Read-backs of earlier
 * steps that have completed are consumed at the start of a step: every
 * expert of that step's cache that has neither landed nor is in flight is
 * copied from pinned host memory on stage_stream (moe_stage_experts into
 * dev_w_*), and lands in the resident set when its event has completed (a
 * later step), so copies overlap the steps that keep running on the old
 * set.  An evicted expert loses its landed status, so a later admission
 * copies it again.  Under MOE_MISS_EXACT the layer instead waits for its
 * misses: the host reads the fetch mask (synchronising), misses already in
 * flight are waited for on the GPU (they landed in time for the layer), the
 * others are copied at once and waited for (a stall).
 * The caller creates the events (cudaEvent_t as void*, timing disabled is
 * fine) and the buffers, zeroes the struct's state fields, sets the
 * configuration and calls moe_cache_start once; the struct then carries the
 * pipeline's state between steps.  One pipeline per layer; not thread-safe. */
#define MOE_CACHE_RING 16
#define MOE_CACHE_FLIGHTS 8
typedef struct {
    /* configuration */
    int capacity;                          /* experts in the cache */
    float decay;                           /* heat decay per step, in [0, 1] */
    int max_flight_experts;                /* experts being copied at once, at most (<= 0: no bound) */
    /* caller-owned resources */
    uint64_t* host_ring;                   /* pinned host uint64[MOE_CACHE_RING * 4] */
    void* step_events[MOE_CACHE_RING];     /* one per ring entry */
    void* copy_events[MOE_CACHE_FLIGHTS];  /* one per copy batch in flight */
    uint64_t* dev_masks;                   /* device uint64[4]: cache, (reserved), resident, admit */
    float* dev_heat;                       /* device float32[N] */
    int32_t* dev_stats;                    /* device int32[4] or NULL: moe_cache_update's counters */
    /* state (kept by the library) */
    long long step, consumed;
    uint64_t landed, in_flight;
    uint64_t flight_mask[MOE_CACHE_FLIGHTS];
    /* totals since moe_cache_start */
    long long staged_experts, staged_bytes;    /* admission and stall copies queued */
    long long in_time_experts;                 /* EXACT misses that were already in flight or landed */
    long long stall_experts, stall_steps;      /* EXACT misses copied on demand, and the steps with any */
    uint64_t* dev_ring;                        /* the ring's device address if mapped, else NULL (set by start) */
} moe_cache_pipe;

/* Reset the pipeline's state: cache = landed = resident = start_set (experts
 * preloaded on the device), heat = 0, admit = 0, counters zeroed; queued on
 * `stream`.  Errors: INVALID_ARG (NULL resources, capacity < 0, decay
 * outside [0, 1], start_set with experts >= N), CUDA. */
moe_status moe_cache_start(const moe_dims* dims, moe_cache_pipe* pipe, uint64_t start_set, void* stream);

/* One decode step of the pipeline (see above): args as for
 * moe_layer_forward (its resident / n_resident are replaced by the
 * pipeline's), outs its outputs; host_w_* pinned host copies and dev_w_*
 * device homes of the N routed experts.  Errors: those of the stages, CUDA,
 * STAGING. */
moe_status moe_cache_step(const moe_dims* dims, const moe_layer_args* args, const moe_layer_outputs* outs,
                          moe_cache_pipe* pipe, const void* const* host_w_gate, const void* const* host_w_up,
                          const void* const* host_w_down, void* const* dev_w_gate, void* const* dev_w_up,
                          void* const* dev_w_down, void* ws, size_t ws_bytes, void* stream, void* stage_stream);

/* Wait for every copy in flight and every queued read-back, and fold them
 * into the state (for the end of a run or a test). */
moe_status moe_cache_drain(const moe_dims* dims, moe_cache_pipe* pipe, const void* const* host_w_gate,
                           const void* const* host_w_up, const void* const* host_w_down, void* const* dev_w_gate,
                           void* const* dev_w_up, void* const* dev_w_down, void* stage_stream);

/* Synchronise `stream`, read and clear the device error word of `ws`.
 * *device_status receives MOE_OK or the first error a kernel recorded;
 * *detail (may be NULL) a code-specific detail (token, expert or stage). */
moe_status moe_check(void* ws, void* stream, moe_status* device_status, int32_t* detail);

/* Text of the last MOE_ERR_CUDA on this host thread: the failing call and
 * the CUDA error name and message ("" if none).  Valid until the next call
 * on this thread. */
const char* moe_last_error_detail(void);

/* Total number of kernel launches this library has queued since it was
 * loaded (all threads).  Read it before and after a region to count the
 * kernels launched inside it. */
uint64_t moe_launch_total(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
