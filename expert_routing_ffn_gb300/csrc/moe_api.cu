// C ABI of the MoE layer (include/moe.h): argument checks, workspace layout,
// expert table, and the launch sequence of each stage.
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "../../include/moe_testing.h"
#include "tma.h"

using namespace moe;

static thread_local char g_launch_note[256] = "";

namespace moe {

cudaError_t note_launch(const void* kernel, int threads, size_t dyn_smem, cudaError_t e) {
    if (e == cudaSuccess) return e;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kernel) == cudaSuccess)
        std::snprintf(g_launch_note, sizeof(g_launch_note),
                      "kernel regs=%d maxThreads=%d staticSmem=%zu maxDynSmem=%d; launch threads=%d "
                      "dynSmem=%zu", fa.numRegs, fa.maxThreadsPerBlock, fa.sharedSizeBytes,
                      fa.maxDynamicSharedSizeBytes, threads, dyn_smem);
    return e;
}

cudaError_t allow_max_smem_impl(const void* kernel) {
    static std::mutex mu;
    static std::vector<std::pair<const void*, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (const auto& p : done)
        if (p.first == kernel && p.second == dev) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    // static + dynamic shared memory of one block may not exceed the opt-in size
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)fa.sharedSizeBytes);
    if (e == cudaSuccess) done.emplace_back(kernel, dev);
    return e;
}

}  // namespace moe

namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_fail_copies_after{-1};

inline void count(int n = 1) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

}  // namespace

namespace moe {
void note_launches(int n) { count(n); }
}  // namespace moe

namespace {

inline cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }


#define MOE_TRY(expr)                                      \
    do {                                                   \
        moe_status _st = (expr);                           \
        if (_st != MOE_OK) return _st;                     \
    } while (0)

thread_local char g_detail[512] = "";

moe_status record_cuda(cudaError_t e, const char* what) {
    std::snprintf(g_detail, sizeof(g_detail), "%s: %s (%s)%s%s", what, cudaGetErrorName(e),
                  cudaGetErrorString(e), g_launch_note[0] ? "; " : "", g_launch_note);
    g_launch_note[0] = 0;
    return MOE_ERR_CUDA;
}

#define MOE_CUDA(expr)                                     \
    do {                                                   \
        cudaError_t _e = (expr);                           \
        if (_e != cudaSuccess) return record_cuda(_e, #expr); \
    } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_dims(const moe_dims* D) {
    if (!D) return MOE_ERR_INVALID_ARG;
    if (D->T < 0 || D->d <= 0 || D->N <= 0 || D->k <= 0 || D->I <= 0 || D->n_shared < 0 ||
        D->r < 0 || D->delta_max < 0)
        return MOE_ERR_INVALID_ARG;
    if (D->n_shared > 0 && D->I_shared <= 0) return MOE_ERR_INVALID_ARG;
    if (D->wtype != MOE_DTYPE_BF16 && D->wtype != MOE_DTYPE_F32) return MOE_ERR_UNSUPPORTED;
    if (D->N > kMaxExperts || D->k > kMaxTopK || D->k > D->N) return MOE_ERR_UNSUPPORTED;
    if (D->delta_max > D->N - D->k) return MOE_ERR_INVALID_ARG;
    if (D->d % 256 != 0) return MOE_ERR_UNSUPPORTED;
    if (D->wtype == MOE_DTYPE_BF16 && D->d > 4096) return MOE_ERR_UNSUPPORTED;
    if (D->wtype == MOE_DTYPE_F32 && D->d > 1024) return MOE_ERR_UNSUPPORTED;
    if (D->r > 64) return MOE_ERR_UNSUPPORTED;
    if (D->n_shared > kMaxShared) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status check_ws(const moe_dims* D, void* ws, size_t ws_bytes) {
    if (!ws) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) % kAlign) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < ws_layout(*D).total) return MOE_ERR_CAPACITY;
    return MOE_OK;
}

int sm_count() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

int gemv_grid(const moe_dims* D) {
    return gemv_grid_for(D->d, D->wtype == MOE_DTYPE_BF16, sm_count());
}

bool bf16(const moe_dims* D) { return D->wtype == MOE_DTYPE_BF16; }

int tcd_grid() { return sm_count() < kTcdMaxCtas ? sm_count() : kTcdMaxCtas; }

// A second stream per device on which moe_layer_forward runs the LoRE z
// kernel beside the expert FFN (fork and join by events; under stream capture
// this becomes a parallel branch of the graph).  Created on first use.
struct SideStream {
    std::mutex mu;
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

SideStream* side_stream() {
    static std::mutex mu;
    static SideStream per_dev[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    SideStream& sd = per_dev[dev];
    if (!sd.s) {
        if (cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        if (cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess)
            return nullptr;
    }
    return &sd;
}

// Argument checks and launch arguments of the routing stages (T > 0), shared
// by the stage-wise calls and the fused front end of moe_layer_forward.
moe_status prep_route(const moe_dims* dims, const void* x, const void* w_router, const float* router_bias,
                      const void* x_pre, const void* w_prefetch, const float* w_ord, const float* theta,
                      float tau, int n_resident, int32_t* topk_idx, float* topk_gate, float* router_prob,
                      int32_t* delta_hat, uint64_t* prefetch_mask, int32_t* delta_star,
                      uint64_t* batch_resident, void* ws, LogitsArgs& la, RouteSelectArgs& ra) {
    if (!x || !w_router || !topk_idx || !topk_gate || !router_prob || !delta_hat || !prefetch_mask)
        return MOE_ERR_INVALID_ARG;
    const bool has_pref = w_prefetch != nullptr;
    if (has_pref && (!w_ord || !theta || !(tau > 0.f && tau < 1.f))) return MOE_ERR_INVALID_ARG;
    if (n_resident > 0 && (!has_pref || !batch_resident || n_resident > dims->N)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_router) || (x_pre && !aligned16(x_pre)) ||
        (w_prefetch && !aligned16(w_prefetch)))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*dims);
    la.x = x; la.x_pre = x_pre; la.w_router = w_router; la.w_prefetch = w_prefetch;
    la.bias = router_bias; la.w_ord = w_ord; la.T = dims->T; la.d = dims->d; la.N = dims->N;
    la.has_prefetch = has_pref; la.bf16 = bf16(dims);
    la.logits_r = ws_at<float>(ws, L.logits_r); la.logits_p = ws_at<float>(ws, L.logits_p);
    la.score = ws_at<float>(ws, L.score);
    la.part = ws_at<float>(ws, L.route_part); la.sms = sm_count(); la.err = ws_at<DevError>(ws, L.err);
    ra.logits_r = la.logits_r; ra.logits_p = la.logits_p; ra.score = la.score; ra.theta = theta;
    ra.logit_tau = has_pref ? (float)std::log((double)tau / (1.0 - (double)tau)) : 0.f;
    ra.T = dims->T; ra.N = dims->N; ra.k = dims->k; ra.delta_max = dims->delta_max;
    ra.has_prefetch = has_pref; ra.topk_idx = topk_idx; ra.topk_gate = topk_gate;
    ra.router_prob = router_prob; ra.delta_hat = delta_hat; ra.prefetch_mask = prefetch_mask;
    ra.delta_star = delta_star; ra.qp = n_resident > 0 ? ws_at<float>(ws, L.qp) : nullptr;
    return MOE_OK;
}

moe_status prep_select(const moe_dims* dims, const float* router_prob, const int32_t* topk_idx,
                       const uint64_t* prefetch_mask, const uint64_t* resident, int policy, float gamma,
                       const int32_t* delta_hat, const int32_t* delta_star, int32_t* final_idx,
                       float* final_gate, int32_t* final_kind, uint64_t* fetch_mask, int32_t* counters,
                       void* ws, SelectArgs& a) {
    // HETERO only through moe_select_hetero (its callers check the rest)
    if (policy < MOE_MISS_EXACT || policy > MOE_MISS_HETERO) return MOE_ERR_INVALID_ARG;
    if ((policy == MOE_MISS_LORE || policy == MOE_MISS_HYBRID) && dims->r <= 0) return MOE_ERR_INVALID_ARG;
    if (!router_prob || !topk_idx || !final_idx || !final_gate || !final_kind) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*dims);
    a.router_prob = router_prob; a.topk_idx = topk_idx; a.prefetch_mask = prefetch_mask;
    a.resident = resident; a.policy = policy; a.gamma = gamma; a.delta_hat = delta_hat;
    a.delta_star = delta_star; a.T = dims->T; a.N = dims->N; a.k = dims->k;
    a.renorm = dims->renorm_topk; a.final_idx = final_idx; a.final_gate = final_gate;
    a.final_kind = final_kind; a.fetch_mask = fetch_mask; a.counters = counters;
    a.err = ws_at<DevError>(ws, L.err);
    return MOE_OK;
}

moe_status prep_permute(const moe_dims* dims, const int32_t* final_idx, const int32_t* final_kind,
                        int32_t* expert_offsets, int32_t* perm, int32_t* inv_perm, void* ws, PermuteArgs& a,
                        PlanArgs& pa) {
    if (!expert_offsets || !final_idx || !final_kind || !perm || !inv_perm) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*dims);
    DevError* err = ws_at<DevError>(ws, L.err);
    a.final_idx = final_idx; a.final_kind = final_kind; a.n_slots = dims->T * dims->k; a.N = dims->N;
    a.expert_offsets = expert_offsets; a.perm = perm; a.inv_perm = inv_perm; a.err = err;
    pa.expert_offsets = expert_offsets; pa.T = dims->T; pa.N = dims->N; pa.n_shared = dims->n_shared;
    pa.I = dims->I; pa.I_shared = dims->I_shared;
    if (tcd_usable(*dims)) {  // the plan of the decode tensor-core path
        pa.rg = tcd_rows(dims->T); pa.G = tcd_grid(); pa.p_align = 16;
    } else {
        pa.rg = gemv_rows(*dims); pa.G = gemv_grid(dims); pa.p_align = 1;
    }
    pa.max_segs = L.max_segs; pa.max_partial_rows = L.max_partial_rows;
    pa.hdr = ws_at<PlanHeader>(ws, L.plan_hdr); pa.segs = ws_at<Seg>(ws, L.segs);
    pa.seg_first = ws_at<int32_t>(ws, L.seg_first); pa.err = err; pa.d = dims->d;
    pa.tc_plan = use_tc(*dims) ? ws_at<TcPlan>(ws, L.tc_plan) : nullptr;
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported dimensions or type";
        case MOE_ERR_CAPACITY: return "capacity exceeded (buffer too small or available set < k)";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_STAGING: return "expert staging copy failed";
        case MOE_ERR_TIMEOUT: return "bounded device wait timed out";
        case MOE_ERR_DEVICE_INDEX: return "expert or slot index out of range";
    }
    return "unknown status";
}

uint64_t moe_launch_total(void) { return g_launches.load(); }

const char* moe_last_error_detail(void) { return g_detail; }

moe_status moe_workspace_size(const moe_dims* dims, size_t* bytes) {
    MOE_TRY(check_dims(dims));
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = ws_layout(*dims).total;
    return MOE_OK;
}

moe_status moe_expert_table_size(const moe_dims* dims, size_t* bytes) {
    MOE_TRY(check_dims(dims));
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = (size_t)(dims->N + dims->n_shared) * sizeof(ExpertEntry);
    return MOE_OK;
}

moe_status moe_expert_table_init(const moe_dims* dims, const void* const* host_w_gate,
                                 const void* const* host_w_up, const void* const* host_w_down,
                                 const void* const* host_sh_gate, const void* const* host_sh_up,
                                 const void* const* host_sh_down, void* table, size_t table_bytes,
                                 void* stream) {
    MOE_TRY(check_dims(dims));
    const int N = dims->N, ns = dims->n_shared;
    if (!table || !host_w_gate || !host_w_up || !host_w_down) return MOE_ERR_INVALID_ARG;
    if (ns > 0 && (!host_sh_gate || !host_sh_up || !host_sh_down)) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(table) % 64) return MOE_ERR_INVALID_ARG;
    if (table_bytes < (size_t)(N + ns) * sizeof(ExpertEntry)) return MOE_ERR_CAPACITY;
    std::vector<ExpertEntry> h((size_t)(N + ns));
    std::memset(h.data(), 0, h.size() * sizeof(ExpertEntry));
    for (int e = 0; e < N + ns; ++e) {
        const bool sh = e >= N;
        const void* const* src[3] = {sh ? host_sh_gate : host_w_gate, sh ? host_sh_up : host_w_up,
                                     sh ? host_sh_down : host_w_down};
        const int idx = sh ? e - N : e;
        ExpertEntry& E = h[(size_t)e];
        E.I = sh ? dims->I_shared : dims->I;
        for (int m = 0; m < 3; ++m) {
            const void* p = src[m][idx];
            if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
            E.w[m] = p;
        }
        if (bf16(dims)) MOE_TRY(encode_expert_tmaps(E, dims->d));
    }
    MOE_CUDA(cudaMemcpyAsync(table, h.data(), h.size() * sizeof(ExpertEntry), cudaMemcpyHostToDevice,
                             S(stream)));
    MOE_CUDA(cudaStreamSynchronize(S(stream)));
    return MOE_OK;
}

moe_status moe_route(const moe_dims* dims, const void* x, const void* w_router,
                     const float* router_bias, const void* x_pre, const void* w_prefetch,
                     const float* w_ord, const float* theta, float tau, int n_resident,
                     int32_t* topk_idx, float* topk_gate, float* router_prob, int32_t* delta_hat,
                     uint64_t* prefetch_mask, int32_t* delta_star, uint64_t* batch_resident,
                     void* ws, size_t ws_bytes, void* stream) {
    MOE_TRY(check_dims(dims));
    MOE_TRY(check_ws(dims, ws, ws_bytes));
    if (dims->T == 0) return MOE_OK;  // empty batch: nothing to do, buffers may be empty
    LogitsArgs la;
    RouteSelectArgs ra;
    MOE_TRY(prep_route(dims, x, w_router, router_bias, x_pre, w_prefetch, w_ord, theta, tau, n_resident,
                       topk_idx, topk_gate, router_prob, delta_hat, prefetch_mask, delta_star, batch_resident,
                       ws, la, ra));
    MOE_CUDA(launch_logits(la, S(stream)));
    count();
    MOE_CUDA(launch_route_select(ra, S(stream)));
    count();
    if (n_resident > 0) {
        MOE_CUDA(launch_batch_resident(ra.qp, dims->T, dims->N, n_resident, batch_resident,
                                       ws_at<float>(ws, ws_layout(*dims).res_part), S(stream)));
        count();
    }
    return MOE_OK;
}

moe_status moe_select_resident(const moe_dims* dims, const float* router_prob,
                               const int32_t* topk_idx, const uint64_t* prefetch_mask,
                               const uint64_t* resident, int policy, float gamma,
                               const int32_t* delta_hat, const int32_t* delta_star,
                               int32_t* final_idx, float* final_gate, int32_t* final_kind,
                               uint64_t* fetch_mask, int32_t* counters, void* ws, size_t ws_bytes,
                               void* stream) {
    MOE_TRY(check_dims(dims));
    MOE_TRY(check_ws(dims, ws, ws_bytes));
    if (policy < MOE_MISS_EXACT || policy > MOE_MISS_HYBRID) return MOE_ERR_INVALID_ARG;
    if ((policy == MOE_MISS_LORE || policy == MOE_MISS_HYBRID) && dims->r <= 0) return MOE_ERR_INVALID_ARG;
    if (counters) MOE_CUDA(cudaMemsetAsync(counters, 0, MOE_NUM_COUNTERS * sizeof(int32_t), S(stream)));
    if (fetch_mask) MOE_CUDA(cudaMemsetAsync(fetch_mask, 0, sizeof(uint64_t), S(stream)));
    if (dims->T == 0) return MOE_OK;
    SelectArgs a;
    MOE_TRY(prep_select(dims, router_prob, topk_idx, prefetch_mask, resident, policy, gamma, delta_hat,
                        delta_star, final_idx, final_gate, final_kind, fetch_mask, counters, ws, a));
    MOE_CUDA(launch_select_resident(a, S(stream)));
    count();
    return MOE_OK;
}

moe_status moe_select_hetero(const moe_dims* dims, const float* router_prob, const int32_t* topk_idx,
                             const uint64_t* prefetch_mask, const uint64_t* resident, float gamma,
                             int fetch_min_rows, const int32_t* delta_hat, const int32_t* delta_star,
                             int32_t* final_idx, float* final_gate, int32_t* final_kind, int32_t* perm,
                             int32_t* inv_perm, uint64_t* fetch_mask, uint64_t* cpu_mask, int32_t* counters,
                             void* ws, size_t ws_bytes, void* stream) {
    MOE_TRY(check_dims(dims));
    MOE_TRY(check_ws(dims, ws, ws_bytes));
    if (fetch_min_rows < 1 || !(gamma >= 0.f) || (gamma > 0.f && dims->r <= 0) || !perm || !inv_perm)
        return MOE_ERR_INVALID_ARG;
    if (counters) MOE_CUDA(cudaMemsetAsync(counters, 0, MOE_NUM_COUNTERS * sizeof(int32_t), S(stream)));
    if (fetch_mask) MOE_CUDA(cudaMemsetAsync(fetch_mask, 0, sizeof(uint64_t), S(stream)));
    if (cpu_mask) MOE_CUDA(cudaMemsetAsync(cpu_mask, 0, sizeof(uint64_t), S(stream)));
    if (dims->T == 0) return MOE_OK;
    SelectArgs a;
    MOE_TRY(prep_select(dims, router_prob, topk_idx, prefetch_mask, resident, MOE_MISS_HETERO, gamma, delta_hat,
                        delta_star, final_idx, final_gate, final_kind, nullptr, counters, ws, a));
    MOE_CUDA(launch_select_resident(a, S(stream)));
    count();
    MOE_CUDA(launch_hetero_decide(final_idx, final_kind, dims->T * dims->k, dims->N, fetch_min_rows, fetch_mask,
                                  cpu_mask, perm, inv_perm, counters, S(stream)));
    count();
    return MOE_OK;
}

moe_status moe_stage_experts(const moe_dims* dims, uint64_t host_fetch_mask,
                             const void* const* host_w_gate, const void* const* host_w_up,
                             const void* const* host_w_down, void* const* dev_w_gate,
                             void* const* dev_w_up, void* const* dev_w_down, void* stage_stream,
                             void* done_event, size_t* bytes) {
    MOE_TRY(check_dims(dims));
    if (!host_w_gate || !host_w_up || !host_w_down || !dev_w_gate || !dev_w_up || !dev_w_down ||
        !done_event || !bytes)
        return MOE_ERR_INVALID_ARG;
    const uint64_t vm = dims->N >= 64 ? ~0ull : ((1ull << dims->N) - 1ull);
    if (host_fetch_mask & ~vm) return MOE_ERR_INVALID_ARG;
    const size_t mat = (size_t)dims->I * dims->d * (bf16(dims) ? 2 : 4);
    size_t queued = 0;
    int fail_after = g_fail_copies_after.load();
    int n_copies = 0;
    for (int e = 0; e < dims->N; ++e) {
        if (!((host_fetch_mask >> e) & 1)) continue;
        const void* src[3] = {host_w_gate[e], host_w_up[e], host_w_down[e]};
        void* dst[3] = {dev_w_gate[e], dev_w_up[e], dev_w_down[e]};
        for (int m = 0; m < 3; ++m) {
            if (!src[m] || !dst[m]) { *bytes = queued; return MOE_ERR_INVALID_ARG; }
            if (fail_after >= 0 && n_copies >= fail_after) { *bytes = queued; return MOE_ERR_STAGING; }
            if (cudaMemcpyAsync(dst[m], src[m], mat, cudaMemcpyHostToDevice, S(stage_stream)) !=
                cudaSuccess) {
                *bytes = queued;
                return MOE_ERR_STAGING;
            }
            ++n_copies;
            queued += mat;
        }
    }
    *bytes = queued;
    if (cudaEventRecord(reinterpret_cast<cudaEvent_t>(done_event), S(stage_stream)) != cudaSuccess)
        return MOE_ERR_STAGING;
    return MOE_OK;
}

// test hook: make the n-th and later copies of moe_stage_experts fail (-1: off)
void moe_testing_fail_copies_after(int n) { g_fail_copies_after.store(n); }

void moe_testing_set_tc_pairs(int mode) { set_tc_pairs(mode); }

moe_status moe_testing_wait_timeout(void* ws, size_t ws_bytes, void* stream) {
    if (!ws || ws_bytes < kAlign || reinterpret_cast<uintptr_t>(ws) % kAlign) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_wait_timeout_probe(static_cast<DevError*>(ws), S(stream)));
    count();
    return MOE_OK;
}

moe_status moe_permute(const moe_dims* dims, const int32_t* final_idx, const int32_t* final_kind,
                       int32_t* expert_offsets, int32_t* perm, int32_t* inv_perm, void* ws,
                       size_t ws_bytes, void* stream) {
    MOE_TRY(check_dims(dims));
    MOE_TRY(check_ws(dims, ws, ws_bytes));
    if (!expert_offsets) return MOE_ERR_INVALID_ARG;
    if (dims->T == 0) {
        MOE_CUDA(cudaMemsetAsync(expert_offsets, 0, (dims->N + 1) * sizeof(int32_t), S(stream)));
        return MOE_OK;
    }
    PermuteArgs a;
    PlanArgs pa;
    MOE_TRY(prep_permute(dims, final_idx, final_kind, expert_offsets, perm, inv_perm, ws, a, pa));
    const WsLayout L = ws_layout(*dims);
    MOE_CUDA(launch_permute(a, pa, ws_at<int32_t>(ws, L.perm_counts), S(stream)));
    count();
    return MOE_OK;
}

}  // extern "C"

namespace {

// The expert FFN; reduce = false leaves the partial rows of the GEMV and
// decode tensor-core paths unsummed (moe_layer_forward's fused epilogue sums
// them).  The tensor-core prefill path writes y_perm / y_shared directly.
moe_status expert_ffn_impl(const moe_dims* dims, const void* x, const void* table,
                           const int32_t* expert_offsets, const int32_t* perm, float keep_frac,
                           float* y_perm, float* y_shared, void* ws, size_t ws_bytes, void* stream,
                           bool reduce, bool prefetch_shared = false) {
    MOE_TRY(check_dims(dims));
    MOE_TRY(check_ws(dims, ws, ws_bytes));
    if (!(keep_frac > 0.f && keep_frac <= 1.f)) return MOE_ERR_INVALID_ARG;
    const bool floe = keep_frac < 1.f;
    // FloE sparsity runs on the decode (GEMV) path for bf16 layers
    if (floe && (use_tc(*dims) || !bf16(dims))) return MOE_ERR_UNSUPPORTED;
    if (dims->T == 0) return MOE_OK;
    if (!x || !table || !expert_offsets || !perm || !y_perm) return MOE_ERR_INVALID_ARG;
    if (dims->n_shared > 0 && !y_shared) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || reinterpret_cast<uintptr_t>(table) % 64) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*dims);
    if (use_tc(*dims)) {
        // the epilogue writes y_perm / y_shared with TMA stores
        if (!aligned16(y_perm) || (y_shared && !aligned16(y_shared))) return MOE_ERR_INVALID_ARG;
        TcLaunch t;
        t.x = x; t.perm = perm; t.expert_offsets = expert_offsets;
        t.table = static_cast<const ExpertEntry*>(table); t.plan = ws_at<TcPlan>(ws, L.tc_plan);
        t.x_perm = ws_at<void>(ws, L.x_perm); t.h_routed = ws_at<void>(ws, L.h_routed);
        t.h_shared = ws_at<void>(ws, L.h_shared); t.y_perm = y_perm; t.y_shared = y_shared;
        t.dep = ws_at<int>(ws, L.tc_dep);
        t.n_dep = (int)((dims->T + dims->T * dims->k) / 128 + dims->N + 4);
        t.T = dims->T; t.d = dims->d; t.N = dims->N; t.k = dims->k; t.I = dims->I;
        t.I_shared = dims->I_shared; t.n_shared = dims->n_shared; t.rows_cap = dims->T * dims->k;
        t.grid = sm_count(); t.err = ws_at<DevError>(ws, L.err);
        MOE_CUDA(launch_tc_ffn(t, S(stream)));
        count(2);
        return MOE_OK;
    }
    if (!floe && tcd_usable(*dims)) {
        // decode-size batch on the tensor cores (plan built by moe_permute)
        TcdLaunch t;
        t.x = x; t.perm = perm; t.expert_offsets = expert_offsets;
        t.table = static_cast<const ExpertEntry*>(table);
        t.hdr = ws_at<PlanHeader>(ws, L.plan_hdr); t.segs = ws_at<Seg>(ws, L.segs);
        t.x_perm = ws_at<void>(ws, L.x_perm); t.partial = ws_at<float>(ws, L.partial);
        t.T = dims->T; t.d = dims->d; t.N = dims->N; t.k = dims->k; t.rows_cap = dims->T * dims->k;
        t.nt = tcd_rows(dims->T); t.grid = tcd_grid(); t.u_out = nullptr; t.I = dims->I;
        t.err = ws_at<DevError>(ws, L.err); t.prefetch_shared = prefetch_shared ? dims->n_shared : 0;
        MOE_CUDA(launch_tcd_ffn(t, S(stream)));
        count(t.nt == 32 ? 2 : 1);  // + the row gather for 32-row segments
        if (!reduce) return MOE_OK;
        GemvReduceArgs r;
        r.hdr = t.hdr; r.segs = t.segs; r.seg_first = ws_at<int32_t>(ws, L.seg_first);
        r.expert_offsets = expert_offsets; r.partial = t.partial; r.d = dims->d; r.N = dims->N;
        r.n_shared = dims->n_shared; r.T = dims->T; r.routed_cap = dims->T * dims->k;
        r.y_perm = y_perm; r.y_shared = y_shared; r.direct = true;
        MOE_CUDA(launch_gemv_reduce(r, S(stream)));
        count();
        return MOE_OK;
    }
    GemvParams p;
    p.x = x; p.d = dims->d; p.N = dims->N; p.topk = dims->k; p.NS = gemv_stages(dims->d, bf16(dims));
    p.perm = perm; p.table = static_cast<const ExpertEntry*>(table);
    p.hdr = ws_at<PlanHeader>(ws, L.plan_hdr); p.segs = ws_at<Seg>(ws, L.segs);
    p.partial = ws_at<float>(ws, L.partial); p.err = ws_at<DevError>(ws, L.err);
    p.floe_u = ws_at<float>(ws, L.floe_u); p.floe_kept = ws_at<uint32_t>(ws, L.floe_kept);
    p.floe_list = ws_at<int32_t>(ws, L.floe_list); p.I = dims->I; p.words = (dims->I + 31) / 32;
    p.up_pass = 0; p.prefetch_shared = prefetch_shared && !floe ? dims->n_shared : 0;
    if (floe) {
        p.NS = gemv_stages(dims->d, bf16(dims), 4);  // the sparse pass: 4 channels per stage
        FloeArgs f;
        f.x = x; f.perm = perm; f.expert_offsets = expert_offsets; f.table = p.table;
        f.d = dims->d; f.I = dims->I; f.N = dims->N; f.topk = dims->k;
        f.m = (int)std::ceil((double)keep_frac * dims->I - 1e-6);
        if (f.m < 1) f.m = 1;
        f.words = p.words; f.rows_cap = dims->T * dims->k;
        f.u = ws_at<float>(ws, L.floe_u); f.kept = ws_at<uint32_t>(ws, L.floe_kept);
        f.list = ws_at<int32_t>(ws, L.floe_list); f.count = ws_at<int32_t>(ws, L.floe_count);
        // the up pass of 4..64 tokens on the decode tensor cores
        f.tc_nt = tcd_shapes(*dims) && dims->T >= kTcdMinTokens ? tcd_rows(dims->T) : 0;
        f.tc_grid = tcd_grid(); f.x_perm = ws_at<void>(ws, L.x_perm); f.T = dims->T;
        PlanArgs pa;
        pa.expert_offsets = expert_offsets; pa.T = dims->T; pa.N = dims->N;
        pa.n_shared = dims->n_shared; pa.I = dims->I; pa.I_shared = dims->I_shared;
        pa.rg = gemv_rows(*dims); pa.G = gemv_grid(dims); pa.p_align = 1; pa.max_segs = L.max_segs;
        pa.max_partial_rows = L.max_partial_rows; pa.d = dims->d;
        pa.hdr = ws_at<PlanHeader>(ws, L.plan_hdr); pa.segs = ws_at<Seg>(ws, L.segs);
        pa.seg_first = ws_at<int32_t>(ws, L.seg_first); pa.err = p.err; pa.tc_plan = nullptr;
        MOE_CUDA(launch_floe_prepare(f, pa, p, gemv_grid(dims), S(stream)));
        count(5);
    }
    if (gemv1_usable(dims->T, dims->d, bf16(dims), floe))
        MOE_CUDA(launch_gemv1(p, gemv_grid(dims), S(stream)));
    else
        MOE_CUDA(launch_gemv(p, gemv_grid(dims), bf16(dims), S(stream), floe, floe));
    count();
    if (!reduce) return MOE_OK;
    GemvReduceArgs r;
    r.hdr = p.hdr; r.segs = p.segs; r.seg_first = ws_at<int32_t>(ws, L.seg_first);
    r.expert_offsets = expert_offsets; r.partial = p.partial; r.d = dims->d; r.N = dims->N;
    r.n_shared = dims->n_shared; r.T = dims->T; r.routed_cap = dims->T * dims->k;
    r.y_perm = y_perm; r.y_shared = y_shared; r.direct = false;
    MOE_CUDA(launch_gemv_reduce(r, S(stream)));
    count();
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_expert_ffn(const moe_dims* dims, const void* x, const void* table,
                          const int32_t* expert_offsets, const int32_t* perm, float keep_frac,
                          float* y_perm, float* y_shared, void* ws, size_t ws_bytes, void* stream) {
    return expert_ffn_impl(dims, x, table, expert_offsets, perm, keep_frac, y_perm, y_shared, ws, ws_bytes,
                           stream, true);
}

const char* moe_expert_ffn_path(const moe_dims* dims, float keep_frac) {
    if (!dims || check_dims(dims) != MOE_OK || !(keep_frac > 0.f && keep_frac <= 1.f)) return "unsupported";
    const bool floe = keep_frac < 1.f;
    if (floe) return use_tc(*dims) || !bf16(dims) ? "unsupported" : "gemv-floe";
    if (use_tc(*dims)) return "tc-prefill";
    if (tcd_usable(*dims)) return "tc-decode";
    if (gemv1_usable(dims->T, dims->d, bf16(dims), false)) return "gemv-1tok";
    return "gemv";
}

moe_status moe_floe_kept_mask(const moe_dims* dims, void* ws, size_t ws_bytes, const uint32_t** kept,
                              int32_t* words_per_row) {
    MOE_TRY(check_dims(dims));
    MOE_TRY(check_ws(dims, ws, ws_bytes));
    if (!kept || !words_per_row) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*dims);
    *kept = ws_at<const uint32_t>(ws, L.floe_kept);
    *words_per_row = (dims->I + 31) / 32;
    return MOE_OK;
}

namespace {

// moe_lore; skip_sum: on the grouped path leave y_lore unwritten (the
// prefill epilogue sums the slots' v rows itself).
moe_status lore_impl(const moe_dims* dims, const void* x, const int32_t* final_idx, const int32_t* final_kind,
                     const float* final_gate, const void* lore_a, const void* lore_b, float* y_lore, void* ws,
                     size_t ws_bytes, void* stream, bool skip_sum) {
    MOE_TRY(check_dims(dims));
    if (dims->r <= 0) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_ws(dims, ws, ws_bytes));
    if (dims->T == 0) return MOE_OK;
    if (!x || !final_idx || !final_kind || !final_gate || !y_lore || !lore_a || !lore_b)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(lore_a)) return MOE_ERR_INVALID_ARG;
    LoreArgs a;
    a.x = x; a.final_idx = final_idx; a.final_kind = final_kind; a.final_gate = final_gate;
    a.A = lore_a; a.B = lore_b; a.T = dims->T; a.d = dims->d; a.k = dims->k; a.r = dims->r;
    const WsLayout L = ws_layout(*dims);
    a.N = dims->N; a.bf16 = bf16(dims); a.y_lore = y_lore;
    a.z = ws_at<float>(ws, L.lore_z); a.err = ws_at<DevError>(ws, L.err);
    // (the workspace holds the grouped path's buffers for these dimensions)
    const bool grouped = lore_grouped_usable(dims->T, dims->d, dims->r, bf16(dims));
    a.g_off = ws_at<int32_t>(ws, L.lore_off); a.g_list = ws_at<int32_t>(ws, L.lore_list);
    a.g_pos = ws_at<int32_t>(ws, L.lore_pos); a.g_counts = ws_at<int32_t>(ws, L.lore_counts);
    a.zp = ws_at<float>(ws, L.lore_zp);
    a.v = grouped ? ws_at<float>(ws, L.lore_v) : nullptr;
    a.skip_sum = grouped && skip_sum;
    MOE_CUDA(launch_lore(a, S(stream)));
    // grouped: slot grouping (2 launches), z, z sum, B z and (unless skipped) the per-token sum
    count(grouped ? (a.skip_sum ? 5 : 6) : 2);
    return MOE_OK;
}

}  // namespace

moe_status moe_lore(const moe_dims* dims, const void* x, const int32_t* final_idx,
                    const int32_t* final_kind, const float* final_gate, const void* lore_a,
                    const void* lore_b, float* y_lore, void* ws, size_t ws_bytes, void* stream) {
    return lore_impl(dims, x, final_idx, final_kind, final_gate, lore_a, lore_b, y_lore, ws, ws_bytes, stream,
                     false);
}

moe_status moe_cache_update(const moe_dims* dims, const int32_t* topk_idx, float decay, int capacity,
                            float* heat, uint64_t* cache_mask, uint64_t* admit_mask, int32_t* stats,
                            void* stream) {
    MOE_TRY(check_dims(dims));
    if (!topk_idx || !heat || !cache_mask) return MOE_ERR_INVALID_ARG;
    if (!(decay >= 0.f && decay <= 1.f) || capacity < 0) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_cache_update(topk_idx, dims->T * dims->k, dims->N, decay, capacity, heat, cache_mask, admit_mask,
                                 stats, S(stream)));
    count();
    return MOE_OK;
}

moe_status moe_prefetch_depth(const moe_dims* dims, int n_ahead, const void* x,
                              const void* const* w_router_ahead, const float* const* bias_ahead, float tau,
                              int d_min, float* logits_ahead, float* conf, int32_t* depth,
                              uint64_t* token_masks, uint64_t* layer_masks, void* ws, size_t ws_bytes,
                              void* stream) {
    MOE_TRY(check_dims(dims));
    MOE_TRY(check_ws(dims, ws, ws_bytes));
    if (n_ahead < 1 || n_ahead > MOE_MAX_AHEAD || d_min < 0 || !std::isfinite(tau)) return MOE_ERR_INVALID_ARG;
    if (!w_router_ahead || !layer_masks) return MOE_ERR_INVALID_ARG;
    for (int j = 0; j < n_ahead; ++j)
        if (!w_router_ahead[j] || !aligned16(w_router_ahead[j])) return MOE_ERR_INVALID_ARG;
    if (dims->T > 0 && (!x || !aligned16(x) || !logits_ahead || !conf || !depth || !token_masks))
        return MOE_ERR_INVALID_ARG;
    if (dims->T == 0 || dims->T > kTcMinTokens)
        MOE_CUDA(cudaMemsetAsync(layer_masks, 0, (size_t)n_ahead * sizeof(uint64_t), S(stream)));
    if (dims->T == 0) return MOE_OK;
    const WsLayout L = ws_layout(*dims);
    const size_t plane = (size_t)dims->T * dims->N;
    if (dims->T <= kTcMinTokens) {
        // decode-size batch: every look-ahead router in one launch (which
        // also zeroes the layer masks)
        MOE_CUDA(launch_lookahead_logits(x, w_router_ahead, bias_ahead, n_ahead, dims->T, dims->d, dims->N,
                                         bf16(dims), logits_ahead, layer_masks, S(stream)));
        count();
    }
    for (int j = 0; j < n_ahead && dims->T > kTcMinTokens; ++j) {
        // look-ahead layer j's router on the current hidden state, through the
        // router GEMM paths (no prefetch router)
        LogitsArgs la;
        la.x = x; la.x_pre = nullptr; la.w_router = w_router_ahead[j]; la.w_prefetch = nullptr;
        la.bias = bias_ahead ? bias_ahead[j] : nullptr; la.w_ord = nullptr;
        la.T = dims->T; la.d = dims->d; la.N = dims->N; la.has_prefetch = 0; la.bf16 = bf16(dims);
        la.logits_r = logits_ahead + (size_t)j * plane;
        la.logits_p = ws_at<float>(ws, L.logits_p); la.score = ws_at<float>(ws, L.score);
        la.part = ws_at<float>(ws, L.route_part); la.sms = sm_count(); la.err = ws_at<DevError>(ws, L.err);
        MOE_CUDA(launch_logits(la, S(stream)));
        count();
    }
    MOE_CUDA(launch_prefetch_depth(logits_ahead, dims->T, dims->N, dims->k, n_ahead, tau, d_min, conf, depth,
                                   token_masks, layer_masks, S(stream)));
    count();
    return MOE_OK;
}

int moe_prefetch_min_depth(double expert_bytes, double link_bytes_per_s, double layer_seconds) {
    if (!(expert_bytes >= 0.0) || !(link_bytes_per_s > 0.0) || !(layer_seconds > 0.0)) return -1;
    const double q = expert_bytes / (link_bytes_per_s * layer_seconds);
    if (!(q <= 2147483647.0)) return -1;
    const double r = std::nearbyint(q);
    if (std::fabs(q - r) <= 1e-9 * std::fmax(1.0, r)) return (int)r;
    return (int)std::ceil(q);
}

moe_status moe_bitslice_pack(int rows, int cols, moe_dtype wtype, const void* w, int transpose,
                             uint32_t* planes, float* scales, void* stream) {
    if (rows <= 0 || cols <= 0 || !w || !planes || !scales) return MOE_ERR_INVALID_ARG;
    if (wtype != MOE_DTYPE_BF16 && wtype != MOE_DTYPE_F32) return MOE_ERR_UNSUPPORTED;
    if ((transpose ? rows : cols) % 32 != 0) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_bitslice_pack(rows, cols, wtype == MOE_DTYPE_BF16, w, transpose, planes, scales, S(stream)));
    count();
    return MOE_OK;
}

size_t moe_bitslice_scratch_size(int d, int I, int T, int slots) {
    if (d <= 0 || I <= 0 || T < 0 || slots <= 0) return 0;
    // h and y_part rows, then the down launch's counters (T x d/16 int32)
    return (size_t)T * slots * ((size_t)I + d) * sizeof(float) + (size_t)T * (d / 16) * sizeof(int32_t);
}

moe_status moe_bitslice_ffn(int d, int I, int N, int n_shared, int bits, moe_dtype xtype, const void* x, int T, int k,
                            const int32_t* idx, const float* gate, const uint32_t* planes_gate,
                            const float* scales_gate, const uint32_t* planes_up, const float* scales_up,
                            const uint32_t* planes_down, const float* scales_down, int accumulate, float* y,
                            void* scratch, size_t scratch_bytes, void* stream) {
    if (d <= 0 || I <= 0 || N <= 0 || n_shared < 0 || T < 0 || k <= 0 || bits < 1 || bits > 8)
        return MOE_ERR_INVALID_ARG;
    if (d % 32 != 0 || I % 32 != 0) return MOE_ERR_INVALID_ARG;
    if (d > 4096 || I > 4096) return MOE_ERR_UNSUPPORTED;
    if ((long long)T * (k + n_shared) > 65535) return MOE_ERR_UNSUPPORTED;  // (token, slot) pairs on grid.y
    if (xtype != MOE_DTYPE_BF16 && xtype != MOE_DTYPE_F32) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!x || !idx || !planes_gate || !scales_gate || !planes_up || !scales_up || !planes_down || !scales_down ||
        !y || !scratch)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(planes_gate) || !aligned16(planes_up) || !aligned16(planes_down) ||
        !aligned16(scratch))
        return MOE_ERR_INVALID_ARG;
    if (scratch_bytes < moe_bitslice_scratch_size(d, I, T, k + n_shared)) return MOE_ERR_CAPACITY;
    BitsliceArgs a;
    a.d = d; a.I = I; a.N = N; a.ns = n_shared; a.T = T; a.k = k; a.bits = bits; a.accumulate = accumulate ? 1 : 0;
    a.idx = idx; a.gate = gate;
    a.planes_gate = planes_gate; a.planes_up = planes_up; a.planes_down = planes_down;
    a.scales_gate = scales_gate; a.scales_up = scales_up; a.scales_down = scales_down;
    a.h = static_cast<float*>(scratch); a.y_part = a.h + (size_t)T * (k + n_shared) * I; a.y = y;
    a.cnt = reinterpret_cast<int*>(a.y_part + (size_t)T * (k + n_shared) * d);
    MOE_CUDA(launch_bitslice_ffn(a, x, xtype == MOE_DTYPE_BF16, sm_count(), S(stream)));
    count(2);
    return MOE_OK;
}

moe_status moe_combine(const moe_dims* dims, const float* y_perm, const int32_t* inv_perm,
                       const float* final_gate, const int32_t* final_kind, const float* y_shared,
                       const float* y_lore, float* out, void* stream) {
    MOE_TRY(check_dims(dims));
    if (dims->T == 0) return MOE_OK;
    if (!y_perm || !inv_perm || !final_gate || !final_kind || !out) return MOE_ERR_INVALID_ARG;
    CombineArgs a;
    a.y_perm = y_perm; a.inv_perm = inv_perm; a.final_gate = final_gate; a.final_kind = final_kind;
    a.y_shared = y_shared; a.y_lore = y_lore; a.T = dims->T; a.d = dims->d; a.k = dims->k; a.out = out;
    MOE_CUDA(launch_combine(a, S(stream)));
    count();
    return MOE_OK;
}

}  // extern "C"

namespace {

// The launch sequence of one layer forward (moe_layer_forward runs it
// directly, or captures it once into a CUDA graph and replays that).
moe_status layer_forward_launch(const moe_dims* dims, const moe_layer_args* A, const moe_layer_outputs* O,
                                void* ws, size_t ws_bytes, void* stream) {
    MOE_TRY(check_dims(dims));
    if (!A || !O) return MOE_ERR_INVALID_ARG;
    if (A->policy == MOE_MISS_HETERO) return MOE_ERR_INVALID_ARG;  // moe_layer_forward_hetero
    const uint64_t* resident = A->n_resident > 0 ? O->batch_resident : A->resident;
    const uint64_t* pref_mask = A->use_prefetch_mask ? O->prefetch_mask : nullptr;
    if (dims->T > 0 && dims->T <= kFrontMaxTokens && dims->T * dims->k <= kFrontMaxSlots) {
        // small batch: routing, selection, resident set, misses and the
        // permutation in one launch (same device code as the stage-wise calls)
        MOE_TRY(check_ws(dims, ws, ws_bytes));
        FrontArgs f;
        MOE_TRY(prep_route(dims, A->x, A->w_router, A->router_bias, A->x_pre, A->w_prefetch, A->w_ord,
                           A->theta, A->tau, A->n_resident, O->topk_idx, O->topk_gate, O->router_prob,
                           O->delta_hat, O->prefetch_mask, O->delta_star, O->batch_resident, ws, f.la, f.ra));
        MOE_TRY(prep_select(dims, O->router_prob, O->topk_idx, pref_mask, resident, A->policy, A->gamma,
                            O->delta_hat, O->delta_star, O->final_idx, O->final_gate, O->final_kind,
                            O->fetch_mask, O->counters, ws, f.sa));
        MOE_TRY(prep_permute(dims, O->final_idx, O->final_kind, O->expert_offsets, O->perm, O->inv_perm, ws,
                             f.pa, f.plan));
        f.n_resident = A->n_resident; f.batch_resident = O->batch_resident;
        f.ticket = ws_at<int>(ws, ws_layout(*dims).ticket) + 1;
        MOE_CUDA(launch_route_front(f, S(stream)));
        count();
    } else {
        MOE_TRY(moe_route(dims, A->x, A->w_router, A->router_bias, A->x_pre, A->w_prefetch, A->w_ord,
                          A->theta, A->tau, A->n_resident, O->topk_idx, O->topk_gate, O->router_prob,
                          O->delta_hat, O->prefetch_mask, O->delta_star, O->batch_resident, ws,
                          ws_bytes, stream));
        MOE_TRY(moe_select_resident(dims, O->router_prob, O->topk_idx, pref_mask, resident,
                                    A->policy, A->gamma, O->delta_hat, O->delta_star, O->final_idx,
                                    O->final_gate, O->final_kind, O->fetch_mask, O->counters, ws,
                                    ws_bytes, stream));
        MOE_TRY(moe_permute(dims, O->final_idx, O->final_kind, O->expert_offsets, O->perm, O->inv_perm,
                            ws, ws_bytes, stream));
    }
    const bool lore = dims->r > 0 && A->lore_a && A->lore_b && O->y_lore;
    if (!use_tc(*dims) && dims->T > 0) {
        // partial-row paths: FFN without its reduction, LoRE z, then one
        // launch for reduction + LoRE B + combine
        const WsLayout L = ws_layout(*dims);
        if (lore) {
            // LoRE z = g A_e x on the side stream, beside the expert FFN
            LoreArgs la;
            la.x = A->x; la.final_idx = O->final_idx; la.final_kind = O->final_kind;
            la.final_gate = O->final_gate; la.A = A->lore_a; la.B = A->lore_b; la.T = dims->T; la.d = dims->d;
            la.k = dims->k; la.r = dims->r; la.N = dims->N; la.bf16 = bf16(dims);
            la.z = ws_at<float>(ws, L.lore_z); la.y_lore = O->y_lore; la.err = ws_at<DevError>(ws, L.err);
            la.skip_sum = false;
            SideStream* sd = side_stream();
            if (!sd) return MOE_ERR_CUDA;
            std::lock_guard<std::mutex> lock(sd->mu);
            MOE_CUDA(cudaEventRecord(sd->fork, S(stream)));
            MOE_CUDA(cudaStreamWaitEvent(sd->s, sd->fork, 0));
            MOE_CUDA(launch_lore_z(la, sd->s));
            count();
            MOE_CUDA(cudaEventRecord(sd->join, sd->s));
            MOE_TRY(expert_ffn_impl(dims, A->x, A->table, O->expert_offsets, O->perm, A->keep_frac, O->y_perm,
                                    O->y_shared, ws, ws_bytes, stream, false, true));
            MOE_CUDA(cudaStreamWaitEvent(S(stream), sd->join, 0));
        } else {
            MOE_TRY(expert_ffn_impl(dims, A->x, A->table, O->expert_offsets, O->perm, A->keep_frac, O->y_perm,
                                    O->y_shared, ws, ws_bytes, stream, false, true));
        }
        EpilogueArgs ea;
        ea.hdr = ws_at<PlanHeader>(ws, L.plan_hdr); ea.segs = ws_at<Seg>(ws, L.segs);
        ea.seg_first = ws_at<int32_t>(ws, L.seg_first); ea.expert_offsets = O->expert_offsets;
        ea.partial = ws_at<float>(ws, L.partial);
        ea.inv_perm = O->inv_perm; ea.final_idx = O->final_idx; ea.final_kind = O->final_kind;
        ea.final_gate = O->final_gate; ea.z = ws_at<float>(ws, L.lore_z); ea.lore_b = lore ? A->lore_b : nullptr;
        ea.T = dims->T; ea.d = dims->d; ea.N = dims->N; ea.k = dims->k; ea.r = dims->r;
        ea.n_shared = dims->n_shared; ea.bf16 = bf16(dims);
        ea.direct = A->keep_frac >= 1.f && tcd_usable(*dims);  // the partials of the decode tensor-core path
        ea.y_perm = O->y_perm; ea.y_shared = O->y_shared; ea.y_lore = O->y_lore; ea.out = O->out;
        if (!ea.out || !ea.y_perm || !O->inv_perm || (dims->n_shared > 0 && !ea.y_shared))
            return MOE_ERR_INVALID_ARG;
        MOE_CUDA(launch_layer_epilogue(ea, S(stream)));
        count();
        return MOE_OK;
    }
    if (dims->T > 0 && (!lore || lore_grouped_usable(dims->T, dims->d, dims->r, bf16(dims)))) {
        // tensor-core prefill: the expert FFN, LoRE grouped by expert (its
        // B_e z rows), then one launch for their per-token sum and the combine
        if (!O->out || !O->inv_perm || !O->final_gate || !O->final_kind || !O->y_perm ||
            (dims->n_shared > 0 && !O->y_shared))
            return MOE_ERR_INVALID_ARG;
        MOE_TRY(moe_expert_ffn(dims, A->x, A->table, O->expert_offsets, O->perm, A->keep_frac, O->y_perm,
                               O->y_shared, ws, ws_bytes, stream));
        if (lore)
            MOE_TRY(lore_impl(dims, A->x, O->final_idx, O->final_kind, O->final_gate, A->lore_a, A->lore_b,
                              O->y_lore, ws, ws_bytes, stream, true));
        const WsLayout L = ws_layout(*dims);
        PrefillEpilogueArgs pe;
        pe.y_perm = O->y_perm; pe.y_shared = dims->n_shared > 0 ? O->y_shared : nullptr;
        pe.inv_perm = O->inv_perm; pe.final_idx = O->final_idx; pe.final_kind = O->final_kind;
        pe.final_gate = O->final_gate;
        pe.lore_v = lore ? ws_at<float>(ws, L.lore_v) : nullptr; pe.g_pos = ws_at<int32_t>(ws, L.lore_pos);
        pe.T = dims->T; pe.d = dims->d; pe.k = dims->k; pe.out = O->out;
        MOE_CUDA(launch_prefill_epilogue(pe, S(stream)));
        count();
        return MOE_OK;
    }
    MOE_TRY(moe_expert_ffn(dims, A->x, A->table, O->expert_offsets, O->perm, A->keep_frac,
                           O->y_perm, O->y_shared, ws, ws_bytes, stream));
    if (lore)
        MOE_TRY(moe_lore(dims, A->x, O->final_idx, O->final_kind, O->final_gate, A->lore_a,
                         A->lore_b, O->y_lore, ws, ws_bytes, stream));
    MOE_TRY(moe_combine(dims, O->y_perm, O->inv_perm, O->final_gate, O->final_kind,
                        dims->n_shared > 0 ? O->y_shared : nullptr, lore ? O->y_lore : nullptr,
                        O->out, stream));
    return MOE_OK;
}

// Instantiated graphs of moe_layer_forward, keyed by the exact bytes of its
// arguments (dims, the layer arguments, the output pointers, the workspace)
// and the device.  A replay reads the same buffers at the same addresses, so
// the values in them may change between calls.
struct GraphEntry {
    int device;
    moe_dims dims;
    moe_layer_args args;
    moe_layer_outputs outs;
    void* ws;
    size_t ws_bytes;
    const void* host_x;  // moe_layer_forward_host: the copies in and out are part of the graph
    float* host_out;
    cudaGraphExec_t exec;
    int launches;
    uint64_t last_use;
};
constexpr int kMaxGraphs = 48;
std::mutex g_graph_mu;
GraphEntry g_graphs[kMaxGraphs];
int g_n_graphs = 0;
uint64_t g_graph_clock = 0;
std::atomic<int> g_graphs_enabled{1};

bool same_call(const GraphEntry& g, int dev, const moe_dims* D, const moe_layer_args* A, const moe_layer_outputs* O,
               void* ws, size_t ws_bytes, const void* host_x, const float* host_out) {
    return g.device == dev && g.ws == ws && g.ws_bytes == ws_bytes && g.host_x == host_x &&
           g.host_out == host_out && !std::memcmp(&g.dims, D, sizeof(moe_dims)) &&
           !std::memcmp(&g.args, A, sizeof(moe_layer_args)) && !std::memcmp(&g.outs, O, sizeof(moe_layer_outputs));
}

// The launch sequence, with the input copied in from host_x first and the
// output copied out to host_out last when those are given.
moe_status layer_forward_with_copies(const moe_dims* D, const moe_layer_args* A, const moe_layer_outputs* O,
                                     void* ws, size_t ws_bytes, void* stream, const void* host_x, float* host_out) {
    cudaStream_t s = S(stream);
    const size_t x_bytes = (size_t)D->T * D->d * (D->wtype == MOE_DTYPE_BF16 ? 2 : 4);
    if (host_x) MOE_CUDA(cudaMemcpyAsync(const_cast<void*>(A->x), host_x, x_bytes, cudaMemcpyHostToDevice, s));
    MOE_TRY(layer_forward_launch(D, A, O, ws, ws_bytes, stream));
    if (host_out)
        MOE_CUDA(cudaMemcpyAsync(host_out, O->out, (size_t)D->T * D->d * sizeof(float), cudaMemcpyDeviceToHost, s));
    return MOE_OK;
}

// Graph replay of one call (see moe_set_graph_replay); plain launches when
// the stream is being captured, is the legacy default stream, or replay is off.
moe_status forward_replayed(const moe_dims* dims, const moe_layer_args* A, const moe_layer_outputs* O, void* ws,
                            size_t ws_bytes, void* stream, const void* host_x, float* host_out);

}  // namespace

extern "C" {

void moe_set_graph_replay(int enabled) { g_graphs_enabled.store(enabled ? 1 : 0); }

moe_status moe_layer_forward(const moe_dims* dims, const moe_layer_args* A, const moe_layer_outputs* O, void* ws,
                             size_t ws_bytes, void* stream) {
    MOE_TRY(check_dims(dims));
    if (!A || !O) return MOE_ERR_INVALID_ARG;
    return forward_replayed(dims, A, O, ws, ws_bytes, stream, nullptr, nullptr);
}

moe_status moe_layer_forward_host(const moe_dims* dims, const moe_layer_args* A, const moe_layer_outputs* O,
                                  const void* host_x, float* host_out, void* ws, size_t ws_bytes, void* stream) {
    MOE_TRY(check_dims(dims));
    if (!A || !O || !A->x || !O->out || (dims->T > 0 && (!host_x || !host_out))) return MOE_ERR_INVALID_ARG;
    if (A->x_pre && A->x_pre != A->x) return MOE_ERR_INVALID_ARG;
    return forward_replayed(dims, A, O, ws, ws_bytes, stream, host_x, host_out);
}

}  // extern "C"

namespace {

moe_status forward_replayed(const moe_dims* dims, const moe_layer_args* A, const moe_layer_outputs* O, void* ws,
                            size_t ws_bytes, void* stream, const void* host_x, float* host_out) {
    cudaStream_t s = S(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    // inside the caller's own capture, or with replay off: plain launches
    if (dims->T == 0 || !g_graphs_enabled.load() || cudaStreamIsCapturing(s, &cap) != cudaSuccess ||
        cap != cudaStreamCaptureStatusNone || s == nullptr)
        return layer_forward_with_copies(dims, A, O, ws, ws_bytes, stream, host_x, host_out);
    int dev = 0;
    MOE_CUDA(cudaGetDevice(&dev));
    {
        std::lock_guard<std::mutex> lock(g_graph_mu);
        for (int i = 0; i < g_n_graphs; ++i) {
            GraphEntry& g = g_graphs[i];
            if (!same_call(g, dev, dims, A, O, ws, ws_bytes, host_x, host_out)) continue;
            g.last_use = ++g_graph_clock;
            MOE_CUDA(cudaGraphLaunch(g.exec, s));
            count(g.launches);
            return MOE_OK;
        }
    }
    // first call with these arguments: capture the launch sequence
    if (!side_stream()) return MOE_ERR_CUDA;  // created outside the capture
    MOE_CUDA(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
    const uint64_t before = g_launches.load();
    const moe_status st = layer_forward_with_copies(dims, A, O, ws, ws_bytes, stream, host_x, host_out);
    const int launches = (int)(g_launches.load() - before);
    cudaGraph_t graph = nullptr;
    const cudaError_t e = cudaStreamEndCapture(s, &graph);
    if (st != MOE_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
    }
    if (e != cudaSuccess) return record_cuda(e, "cudaStreamEndCapture");
    cudaGraphExec_t exec = nullptr;
    const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ei != cudaSuccess) return record_cuda(ei, "cudaGraphInstantiate");
    MOE_CUDA(cudaGraphLaunch(exec, s));  // the capture's launches are counted already
    std::lock_guard<std::mutex> lock(g_graph_mu);
    int slot = g_n_graphs;
    if (g_n_graphs == kMaxGraphs) {  // replace the least recently used
        slot = 0;
        for (int i = 1; i < kMaxGraphs; ++i)
            if (g_graphs[i].last_use < g_graphs[slot].last_use) slot = i;
        cudaGraphExecDestroy(g_graphs[slot].exec);
    } else {
        ++g_n_graphs;
    }
    GraphEntry& g = g_graphs[slot];
    g.device = dev; g.dims = *dims; g.args = *A; g.outs = *O; g.ws = ws; g.ws_bytes = ws_bytes;
    g.host_x = host_x; g.host_out = host_out;
    g.exec = exec; g.launches = launches; g.last_use = ++g_graph_clock;
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_layer_forward_hetero(const moe_dims* dims, const moe_layer_args* A, const moe_layer_outputs* O,
                                    const moe_hetero_cost* cost, const void* const* host_w_gate,
                                    const void* const* host_w_up, const void* const* host_w_down,
                                    void* const* dev_w_gate, void* const* dev_w_up, void* const* dev_w_down,
                                    const moe_hetero_host* H, int n_threads, void* ws, size_t ws_bytes,
                                    void* stream, void* stage_stream, void* stage_event, moe_hetero_stats* stats) {
    using clk = std::chrono::steady_clock;
    MOE_TRY(check_dims(dims));
    MOE_TRY(check_ws(dims, ws, ws_bytes));
    if (!A || !O || !cost || !H || !host_w_gate || !host_w_up || !host_w_down || !dev_w_gate || !dev_w_up ||
        !dev_w_down || !stage_event)
        return MOE_ERR_INVALID_ARG;
    if (A->keep_frac != 1.f || (A->x_pre && A->x_pre != A->x)) return MOE_ERR_INVALID_ARG;
    if (!H->x || !H->final_idx || !H->final_kind || !H->masks || !H->y_rows || !H->scratch ||
        H->scratch_bytes < moe_cpu_experts_scratch_size(dims))
        return MOE_ERR_INVALID_ARG;
    if (!O->out || !O->y_perm || !O->perm || !O->inv_perm || !O->expert_offsets || !O->final_idx ||
        !O->final_kind || !O->final_gate || (dims->n_shared > 0 && !O->y_shared))
        return MOE_ERR_INVALID_ARG;
    const int nmin = moe_hetero_fetch_min_rows(cost);
    if (nmin < 1) return MOE_ERR_INVALID_ARG;
    moe_hetero_stats st;
    std::memset(&st, 0, sizeof(st));
    st.fetch_min_rows = nmin;
    if (stats) *stats = st;
    const int T = dims->T, k = dims->k, d = dims->d;
    if (T == 0) return MOE_OK;
    cudaStream_t s = S(stream);
    const size_t esz = bf16(dims) ? 2 : 4;
    const auto t0 = clk::now();

    // (1) routing and miss handling on the GPU; decisions (and, for small
    //     batches, the hidden state) down to the host
    MOE_TRY(moe_route(dims, A->x, A->w_router, A->router_bias, A->x_pre, A->w_prefetch, A->w_ord, A->theta,
                      A->tau, A->n_resident, O->topk_idx, O->topk_gate, O->router_prob, O->delta_hat,
                      O->prefetch_mask, O->delta_star, O->batch_resident, ws, ws_bytes, stream));
    const uint64_t* resident = A->n_resident > 0 ? O->batch_resident : A->resident;
    const uint64_t* pref_mask = A->use_prefetch_mask ? O->prefetch_mask : nullptr;
    MOE_TRY(moe_select_hetero(dims, O->router_prob, O->topk_idx, pref_mask, resident, A->gamma, nmin, O->delta_hat,
                              O->delta_star, O->final_idx, O->final_gate, O->final_kind, O->perm, O->inv_perm,
                              O->fetch_mask, nullptr, O->counters, ws, ws_bytes, stream));
    const size_t n_slots = (size_t)T * k;
    MOE_CUDA(cudaMemcpyAsync(H->final_idx, O->final_idx, n_slots * 4, cudaMemcpyDeviceToHost, s));
    MOE_CUDA(cudaMemcpyAsync(H->final_kind, O->final_kind, n_slots * 4, cudaMemcpyDeviceToHost, s));
    const size_t x_bytes = (size_t)T * d * esz;
    const bool x_whole = x_bytes <= ((size_t)4 << 20);
    if (x_whole) MOE_CUDA(cudaMemcpyAsync(H->x, A->x, x_bytes, cudaMemcpyDeviceToHost, s));
    MOE_CUDA(cudaStreamSynchronize(s));
    uint64_t fetch = 0, cpu = 0;
    int cpu_slots = 0, lore_slots = 0, cpu_tokens = 0;
    for (int t = 0; t < T; ++t) {
        bool any = false;
        for (int j = 0; j < k; ++j) {
            const int e = H->final_idx[(size_t)t * k + j], kd = H->final_kind[(size_t)t * k + j];
            if (e < 0 || e >= dims->N) continue;
            if (kd == MOE_KIND_FETCH) fetch |= 1ull << e;
            if (kd == MOE_KIND_CPU) { cpu |= 1ull << e; ++cpu_slots; any = true; }
            if (kd == MOE_KIND_LORE) ++lore_slots;
        }
        if (any && !x_whole) {  // large batch: only the rows of tokens with host slots
            MOE_CUDA(cudaMemcpyAsync(static_cast<char*>(H->x) + (size_t)t * d * esz,
                                     static_cast<const char*>(A->x) + (size_t)t * d * esz, d * esz,
                                     cudaMemcpyDeviceToHost, s));
        }
        cpu_tokens += any ? 1 : 0;
    }
    if (!x_whole && cpu_slots) MOE_CUDA(cudaStreamSynchronize(s));
    H->masks[0] = fetch;
    H->masks[1] = cpu;
    st.wait_ms = std::chrono::duration<double, std::milli>(clk::now() - t0).count();

    // (2) fetches on the staging stream; GPU experts, LoRE and shared experts
    //     on `stream`; the host slots on the host cores meanwhile
    if (fetch) {
        size_t nb = 0;
        MOE_TRY(moe_stage_experts(dims, fetch, host_w_gate, host_w_up, host_w_down, dev_w_gate, dev_w_up,
                                  dev_w_down, stage_stream, stage_event, &nb));
        MOE_CUDA(cudaStreamWaitEvent(s, reinterpret_cast<cudaEvent_t>(stage_event), 0));
        st.fetch_bytes = (double)nb;
        st.fetch_experts = __builtin_popcountll(fetch);
    }
    MOE_TRY(moe_permute(dims, O->final_idx, O->final_kind, O->expert_offsets, O->perm, O->inv_perm, ws, ws_bytes,
                        stream));
    MOE_TRY(moe_expert_ffn(dims, A->x, A->table, O->expert_offsets, O->perm, 1.f, O->y_perm, O->y_shared, ws,
                           ws_bytes, stream));
    const bool lore = dims->r > 0 && A->lore_a && A->lore_b && O->y_lore;
    if (lore)
        MOE_TRY(moe_lore(dims, A->x, O->final_idx, O->final_kind, O->final_gate, A->lore_a, A->lore_b, O->y_lore,
                         ws, ws_bytes, stream));
    int32_t n_rows = 0, first = 0;
    const auto th = clk::now();
    MOE_TRY(moe_cpu_experts(dims, H->x, H->final_idx, H->final_kind, host_w_gate, host_w_up, host_w_down,
                            n_threads, H->y_rows, H->scratch, H->scratch_bytes, &n_rows, &first));
    st.host_ms = std::chrono::duration<double, std::milli>(clk::now() - th).count();

    // (3) the host rows into y_perm after the GPU rows, then every slot merged
    if (n_rows)
        MOE_CUDA(cudaMemcpyAsync(O->y_perm + (size_t)first * d, H->y_rows, (size_t)n_rows * d * sizeof(float),
                                 cudaMemcpyHostToDevice, s));
    MOE_TRY(moe_combine(dims, O->y_perm, O->inv_perm, O->final_gate, O->final_kind,
                        dims->n_shared > 0 ? O->y_shared : nullptr, lore ? O->y_lore : nullptr, O->out, stream));
    st.cpu_slots = n_rows;
    st.lore_slots = lore_slots;
    st.cpu_link_bytes = (double)cpu_tokens * d * esz + (double)n_rows * d * sizeof(float);
    if (stats) *stats = st;
    return MOE_OK;
}

moe_status moe_check(void* ws, void* stream, moe_status* device_status, int32_t* detail) {
    if (!ws || !device_status) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(cudaStreamSynchronize(S(stream)));
    DevError h;
    MOE_CUDA(cudaMemcpy(&h, ws, sizeof(int) * 2, cudaMemcpyDeviceToHost));
    *device_status = (moe_status)h.code;
    if (detail) *detail = h.detail;
    MOE_CUDA(cudaMemset(ws, 0, sizeof(int) * 2));
    return MOE_OK;
}

}  // extern "C"
