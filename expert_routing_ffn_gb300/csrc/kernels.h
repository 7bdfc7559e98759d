// Launch interfaces of the kernels (host side of each .cu file).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// On a failed launch: remember the kernel's resource attributes and the
// launch shape for moe_last_error_detail(); returns e.
cudaError_t note_launch(const void* kernel, int threads, size_t dyn_smem, cudaError_t e);

struct LogitsArgs {
    const void *x, *x_pre, *w_router, *w_prefetch;
    const float *bias, *w_ord;
    int T, d, N, has_prefetch;
    bool bf16;
    float *logits_r, *logits_p, *score;
    // tensor-core path (batches of more than kTcMinTokens bf16 tokens): the
    // split-d partial logits (workspace), SM count, device error word
    float* part;
    int sms;
    DevError* err;
};
cudaError_t launch_logits(const LogitsArgs& a, cudaStream_t st);
// router + prefetch-router logits as one tensor-core GEMM (route_tc.cu)
bool route_tc_usable(int T, int d, int N, bool bf16, bool has_prefetch, bool sep_pre);
size_t route_tc_part_bytes(int T, int N);
cudaError_t launch_route_tc(const LogitsArgs& a, float* part, cudaStream_t st);

struct RouteSelectArgs {
    const float *logits_r, *logits_p, *score, *theta;
    float logit_tau;
    int T, N, k, delta_max, has_prefetch;
    int32_t* topk_idx; float* topk_gate; float* router_prob; int32_t* delta_hat;
    uint64_t* prefetch_mask; int32_t* delta_star; float* qp;
};
cudaError_t launch_route_select(const RouteSelectArgs& a, cudaStream_t st);
// part: workspace of 32 x kMaxExperts floats (large batches)
cudaError_t launch_batch_resident(const float* qp, int T, int N, int n_res, uint64_t* out, float* part,
                                  cudaStream_t st);

struct SelectArgs {
    const float* router_prob; const int32_t* topk_idx; const uint64_t* prefetch_mask;
    const uint64_t* resident; int policy; float gamma; const int32_t* delta_hat;
    const int32_t* delta_star; int T, N, k, renorm;
    int32_t* final_idx; float* final_gate; int32_t* final_kind; uint64_t* fetch_mask;
    int32_t* counters; DevError* err;
};
cudaError_t launch_select_resident(const SelectArgs& a, cudaStream_t st);
// heterogeneous path: FETCH -> CPU per expert by the cost threshold, host slots
// placed after the GPU segments of the permutation (one block)
cudaError_t launch_hetero_decide(const int32_t* final_idx, int32_t* final_kind, int n_slots, int N,
                                 int fetch_min_rows, uint64_t* fetch_mask, uint64_t* cpu_mask, int32_t* perm,
                                 int32_t* inv_perm, int32_t* counters, cudaStream_t st);

struct PermuteArgs {
    const int32_t *final_idx, *final_kind;
    int n_slots, N;
    int32_t *expert_offsets, *perm, *inv_perm;
    DevError* err;
};
struct PlanArgs {
    const int32_t* expert_offsets;
    int T, N, n_shared, I, I_shared, rg, G, max_segs, max_partial_rows, d;
    int p_align;      // channels per CTA rounded up to a multiple of this
    PlanHeader* hdr; Seg* segs; int32_t* seg_first; DevError* err;
    TcPlan* tc_plan;  // also built when non-null
};
// permutation + FFN plan in one launch (the last block builds the plan)
// counts: workspace of ceil(n_slots / kPermChunk) * kMaxExperts ints (batches
// of more than 1024 slots)
cudaError_t launch_permute(const PermuteArgs& a, const PlanArgs& plan, int32_t* counts, cudaStream_t st);
// the LoRE slots grouped by expert, stable in slot order (two launches):
// expert_offsets [N + 1], perm = grouped position -> slot, inv_perm = slot ->
// grouped position or -1
cudaError_t launch_group_lore(const PermuteArgs& a, int32_t* counts, cudaStream_t st);

// The routing front end of a small batch (T <= kFrontMaxTokens, T * k <=
// kFrontMaxSlots) in one
// launch: the blocks compute the router / prefetch logits, the last block to
// finish runs selection, the batch resident set (n_resident > 0), miss
// handling (zeroing counters and fetch mask first) and the permutation with
// the FFN plan, with the same device code as the stage-wise kernels.
constexpr int kFrontMaxSlots = 256;
constexpr int kFrontMaxTokens = 64;
struct FrontArgs {
    LogitsArgs la;
    RouteSelectArgs ra;
    int n_resident; uint64_t* batch_resident;
    SelectArgs sa;
    PermuteArgs pa;
    PlanArgs plan;
    int* ticket;
};
cudaError_t launch_route_front(const FrontArgs& a, cudaStream_t st);
// the FFN plan alone
cudaError_t launch_plan_gemv(const PlanArgs& a, cudaStream_t st);

struct GemvParams {
    const void* x;
    int d, N, topk, NS;
    // FloE sparse mode (routed segments with list_off >= 0)
    float* floe_u;                // [rows, I] up projections (written by the up-only pass)
    const uint32_t* floe_kept;    // [rows, words] kept-channel bitsets
    const int32_t* floe_list;     // [N, I] union channel lists
    int I, words;
    int up_pass;                  // 1: every segment is up-only (FloE first pass)
    const int32_t* perm;
    const ExpertEntry* table;
    const PlanHeader* hdr;
    const Seg* segs;
    float* partial;
    DevError* err;
    int prefetch_shared;          // > 0: that many shared experts pulled into L2 before the wait on routing
};
int gemv_stages(int d, bool bf16, int ch = 2);
int gemv_grid_for(int d, bool bf16, int sms);
cudaError_t launch_gemv(const GemvParams& p, int G, bool bf16, cudaStream_t st, bool floe = false,
                        bool sparse = false);
// one-token batches (every segment one row) of dense bf16 layers with d = 1536
// or 2048: one channel per warp, the same plan and partial rows as launch_gemv
bool gemv1_usable(int T, int d, bool bf16, bool floe);
cudaError_t launch_gemv1(const GemvParams& p, int G, cudaStream_t st);

struct FloeArgs {
    const void* x; const int32_t* perm; const int32_t* expert_offsets; const ExpertEntry* table;
    int d, I, N, topk, m, words, rows_cap;
    float* u; uint32_t* kept; int32_t* list; int32_t* count;
    // up pass on the decode tensor cores (tc_nt > 0: its rows per segment,
    // grid, x_perm for 32-row segments), else on the GEMV
    int tc_nt, tc_grid; void* x_perm; int T;
};
// FloE: up-only plan + GEMV pass, selection, unions and the sparse GEMV plan
// (5 launches)
cudaError_t launch_floe_prepare(const FloeArgs& f, const PlanArgs& plan, const GemvParams& gp, int G,
                                cudaStream_t st);

struct GemvReduceArgs {
    const PlanHeader* hdr; const Seg* segs; const int32_t* seg_first; const int32_t* expert_offsets;
    const float* partial; int d, N, n_shared, T, routed_cap;
    float *y_perm, *y_shared;
    bool direct;  // one thread per column (segments of few pieces: decode tensor-core partials)
};
cudaError_t launch_gemv_reduce(const GemvReduceArgs& a, cudaStream_t st);

struct TcLaunch {
    const void* x; const int32_t* perm; const int32_t* expert_offsets; const ExpertEntry* table;
    const TcPlan* plan; void* x_perm; void* h_routed; void* h_shared; float* y_perm; float* y_shared;
    int T, d, N, k, I, I_shared, n_shared, rows_cap, grid; DevError* err;
    int* dep; int n_dep;  // per (segment, row tile) phase-dependency counters (workspace)
};
// tensor-core expert FFN: gather, then one launch of phase 1 (gate/up + SwiGLU)
// and phase 2 (down) tiles
cudaError_t launch_tc_ffn(const TcLaunch& a, cudaStream_t st);
// -1: choose one CTA per tile or CTA pairs by the batch; 0 / 1: force (tests)
void set_tc_pairs(int mode);
// x_perm[pos] = x[perm[pos] / k] for the routed rows (bf16 rows of d values)
cudaError_t launch_gather_rows(const void* x, const int32_t* perm, const int32_t* expert_offsets, int N,
                               int k, int d, int rows_cap, void* x_perm, cudaStream_t st, int* dep = nullptr,
                               int n_dep = 0);

struct TcdLaunch {
    const void* x; const int32_t* perm; const int32_t* expert_offsets; const ExpertEntry* table;
    const PlanHeader* hdr; const Seg* segs; void* x_perm; float* partial;
    int T, d, N, k, rows_cap, nt, grid;
    float* u_out;  // non-NULL: FloE up pass only, u [rows, I] (fp32); no partial rows
    int I;
    DevError* err;
    int prefetch_shared;  // > 0: that many shared experts pulled into L2 before the wait on routing
};
// decode-size expert FFN on the tensor cores: one launch writing the GEMV
// plan's partial rows (summed by launch_gemv_reduce)
cudaError_t launch_tcd_ffn(const TcdLaunch& a, cudaStream_t st);

struct LoreArgs {
    const void* x; const int32_t *final_idx, *final_kind; const float* final_gate;
    const void *A, *B; int T, d, k, r, N; bool bf16; float* z; float* y_lore; DevError* err;
    // batches of more than kTcMinTokens tokens: the LoRE slots grouped by
    // expert (workspace), and the per-slot B_e z rows
    int32_t *g_off, *g_list, *g_pos, *g_counts; float *zp, *v;
    bool skip_sum;  // grouped path: leave y_lore unwritten (launch_prefill_epilogue sums the v rows)
};
cudaError_t launch_lore(const LoreArgs& a, cudaStream_t st);
// whether launch_lore takes the grouped path (given the workspace buffers)
bool lore_grouped_usable(int T, int d, int r, bool bf16);
// z = g A_e x only (the first half of launch_lore)
cudaError_t launch_lore_z(const LoreArgs& a, cudaStream_t st);

struct EpilogueArgs {
    const PlanHeader* hdr; const Seg* segs; const int32_t* seg_first; const int32_t* expert_offsets;
    const float* partial;
    const int32_t *inv_perm, *final_idx, *final_kind; const float* final_gate;
    const float* z; const void* lore_b;  // lore_b NULL: no LoRE term
    int T, d, N, k, r, n_shared; bool bf16;
    float *y_perm, *y_shared, *y_lore, *out;
    bool direct;  // as GemvReduceArgs::direct
};
// partial-row reduction + LoRE B + combine in one launch (moe_layer_forward)
cudaError_t launch_layer_epilogue(const EpilogueArgs& a, cudaStream_t st);

struct PrefillEpilogueArgs {
    const float *y_perm, *y_shared;  // y_shared NULL: no shared experts
    const int32_t *inv_perm, *final_idx, *final_kind; const float* final_gate;
    // LoRE (lore_v NULL: none): the B_e z rows of the grouped slots (lore_v
    // [pos, d], slot -> pos in g_pos, -1 for the other slots)
    const float* lore_v; const int32_t* g_pos;
    int T, d, k;
    float* out;
};
// the tensor-core prefill path's tail of moe_layer_forward: the per-token
// LoRE sum and the combine in one launch
cudaError_t launch_prefill_epilogue(const PrefillEpilogueArgs& a, cudaStream_t st);

// test probe: a bounded wait on an mbarrier nothing arrives on (records
// MOE_ERR_TIMEOUT in err)
cudaError_t launch_wait_timeout_probe(DevError* err, cudaStream_t st);

// persistent expert cache, one decode step (cache.cu)
// bit-sliced expert weights (bitslice.cu)
struct BitsliceArgs {
    int d, I, N, ns, T, k, bits, accumulate;  // ns shared experts: experts N .. N+ns-1, slots k .. k+ns-1
    const int32_t* idx;     // [T, k] expert per routed slot
    const float* gate;      // [T, k] or NULL (1)
    const uint32_t *planes_gate, *planes_up, *planes_down;  // [N][8][R][C/32]
    const float *scales_gate, *scales_up, *scales_down;     // [N][R]
    float* h;               // [T*(k+ns), I] scratch
    float* y_part;          // [T*(k+ns), d] scratch
    float* y;               // [T, d]
    int* cnt;               // [T, d/16] scratch: finished (token, slot) blocks per (token, output block)
};
cudaError_t launch_bitslice_pack(int rows_in, int cols_in, bool bf16, const void* w, int transpose, uint32_t* planes,
                                 float* scales, cudaStream_t st);
cudaError_t launch_bitslice_ffn(const BitsliceArgs& a, const void* x, bool bf16, int sms, cudaStream_t st);
size_t bitslice_table_bytes(int cols);

// confidence-aware look-ahead prefetch depth (lookahead.cu)
constexpr int kMaxAhead = MOE_MAX_AHEAD;
cudaError_t launch_lookahead_logits(const void* x, const void* const* w, const float* const* b, int J, int T, int d,
                                    int N, bool bf16, float* logits, uint64_t* layer_masks, cudaStream_t st);
cudaError_t launch_prefetch_depth(const float* logits, int T, int N, int K, int J, float tau, int d_min,
                                  float* conf, int32_t* depth, uint64_t* tok_masks, uint64_t* layer_masks,
                                  cudaStream_t st);
cudaError_t launch_cache_update(const int32_t* topk_idx, int n_slots, int N, float decay, int capacity, float* heat,
                                uint64_t* cache, uint64_t* admit, int32_t* stats, cudaStream_t st,
                                uint64_t landed = ~0ull, uint64_t* resident = nullptr, uint64_t* readback = nullptr);
// launch counter of moe_launch_total, for launches queued outside moe_api.cu
void note_launches(int n);

struct CombineArgs {
    const float* y_perm; const int32_t* inv_perm; const float* final_gate;
    const int32_t* final_kind; const float *y_shared, *y_lore; int T, d, k; float* out;
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st);

}  // namespace moe
