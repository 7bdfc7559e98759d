// Overlapped expert-cache pipeline for decode loops.
//
// ELMoE-3D (expert-axis elasticity): the experts the router selects most,
// by a heat that decays every step, stay resident and the subset is refreshed
// as the pattern drifts.  SPICE (confidence-aware prefetch): a copy must start
// early enough to land before its layer; D_min = ceil(W_e / (B T_layer))
// steps for one expert.  Here the cache's admissions are copied on a staging
// stream while later steps keep running on the experts already on the device:
// the layer of a step runs on resident = cache & landed, `landed` being the
// experts whose copies have completed (the host learns that from the copies'
// events, without waiting), and the host learns each step's cache from a
// read-back it consumes once that step has finished.  Nothing on the step
// path synchronises the host, except under the EXACT policy, where a step's
// misses must be on the device before its expert FFN (the host reads the
// fetch mask, and any miss not already in flight is a stall).
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace {

inline cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline cudaEvent_t E(void* e) { return reinterpret_cast<cudaEvent_t>(e); }

#define PIPE_TRY(expr)                                 \
    do {                                               \
        moe_status _st = (expr);                       \
        if (_st != MOE_OK) return _st;                 \
    } while (0)

#define PIPE_CUDA(expr)                                \
    do {                                               \
        if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
    } while (0)

uint64_t valid(int N) { return N >= 64 ? ~0ull : ((1ull << N) - 1ull); }

struct Homes {  // host copies and device homes of the routed experts
    const void* const* hg;
    const void* const* hu;
    const void* const* hd;
    void* const* dg;
    void* const* du;
    void* const* dd;
};

// Completed copies: their experts have landed.
void poll_flights(moe_cache_pipe* p) {
    for (int f = 0; f < MOE_CACHE_FLIGHTS; ++f) {
        if (!p->flight_mask[f]) continue;
        if (cudaEventQuery(E(p->copy_events[f])) != cudaSuccess) continue;
        p->landed |= p->flight_mask[f];
        p->in_flight &= ~p->flight_mask[f];
        p->flight_mask[f] = 0;
    }
}

// Copy `want` (experts neither landed nor in flight) on the staging stream
// into a free flight slot, keeping at most max_flight_experts in flight
// (lowest index first; <= 0: no bound).  Returns the slot used (-1: nothing
// queued).
moe_status stage(const moe_dims* D, moe_cache_pipe* p, uint64_t want, const Homes& h, void* stage_stream,
                 int* slot_out) {
    *slot_out = -1;
    want &= ~p->landed & ~p->in_flight & valid(D->N);
    if (p->max_flight_experts > 0) {
        const int room = p->max_flight_experts - __builtin_popcountll(p->in_flight);
        if (room <= 0) return MOE_OK;
        uint64_t take = 0;
        int n = 0;
        for (uint64_t m = want; m && n < room; m &= m - 1, ++n) take |= m & (~m + 1);
        want = take;
    }
    if (!want) return MOE_OK;
    int f = -1;
    for (int i = 0; i < MOE_CACHE_FLIGHTS; ++i)
        if (!p->flight_mask[i]) { f = i; break; }
    if (f < 0) return MOE_OK;  // every flight slot busy: try again next step
    size_t nb = 0;
    PIPE_TRY(moe_stage_experts(D, want, h.hg, h.hu, h.hd, h.dg, h.du, h.dd, stage_stream, p->copy_events[f], &nb));
    p->flight_mask[f] = want;
    p->in_flight |= want;
    p->staged_experts += __builtin_popcountll(want);
    p->staged_bytes += (long long)nb;
    *slot_out = f;
    return MOE_OK;
}

// Fold in a finished step's read-back: evicted experts lose their landed
// status; the step's cache members that are missing get copied.
moe_status consume(const moe_dims* D, moe_cache_pipe* p, long long s, const Homes& h, void* stage_stream) {
    const uint64_t* ring = p->host_ring + (size_t)(s % MOE_CACHE_RING) * 4;
    const uint64_t cache = ring[0];
    p->landed &= cache | p->in_flight;
    int f;
    return stage(D, p, cache, h, stage_stream, &f);
}

moe_status consume_ready(const moe_dims* D, moe_cache_pipe* p, const Homes& h, void* stage_stream) {
    while (p->consumed < p->step) {
        const cudaError_t q = cudaEventQuery(E(p->step_events[p->consumed % MOE_CACHE_RING]));
        if (q == cudaErrorNotReady) break;
        if (q != cudaSuccess) return MOE_ERR_CUDA;
        PIPE_TRY(consume(D, p, p->consumed, h, stage_stream));
        ++p->consumed;
    }
    return MOE_OK;
}

bool pipe_ok(const moe_dims* D, const moe_cache_pipe* p) {
    if (!D || !p || !p->host_ring || !p->dev_masks || !p->dev_heat) return false;
    if (p->capacity < 0 || !(p->decay >= 0.f && p->decay <= 1.f)) return false;
    for (int i = 0; i < MOE_CACHE_RING; ++i)
        if (!p->step_events[i]) return false;
    for (int i = 0; i < MOE_CACHE_FLIGHTS; ++i)
        if (!p->copy_events[i]) return false;
    return true;
}

}  // namespace

extern "C" {

moe_status moe_cache_start(const moe_dims* dims, moe_cache_pipe* p, uint64_t start_set, void* stream) {
    size_t ws = 0;
    PIPE_TRY(moe_workspace_size(dims, &ws));  // validates dims
    if (!pipe_ok(dims, p) || (start_set & ~valid(dims->N))) return MOE_ERR_INVALID_ARG;
    p->step = p->consumed = 0;
    p->landed = start_set;
    p->in_flight = 0;
    for (int f = 0; f < MOE_CACHE_FLIGHTS; ++f) p->flight_mask[f] = 0;
    p->staged_experts = p->staged_bytes = p->in_time_experts = p->stall_experts = p->stall_steps = 0;
    uint64_t* r = p->host_ring;
    std::memset(r, 0, sizeof(uint64_t) * 4 * MOE_CACHE_RING);
    // the cache kernel writes each step's masks into the ring itself when the
    // pinned ring is mapped into the device's address space
    void* dptr = nullptr;
    p->dev_ring = cudaHostGetDevicePointer(&dptr, r, 0) == cudaSuccess ? static_cast<uint64_t*>(dptr) : nullptr;
    cudaGetLastError();  // a ring that is not mapped is not an error: the masks are copied instead
    r[0] = start_set;  // cache
    r[1] = start_set;  // landed
    r[2] = start_set;  // resident
    r[3] = 0;          // admit
    PIPE_CUDA(cudaMemcpyAsync(p->dev_masks, r, 4 * sizeof(uint64_t), cudaMemcpyHostToDevice, S(stream)));
    PIPE_CUDA(cudaMemsetAsync(p->dev_heat, 0, sizeof(float) * (size_t)dims->N, S(stream)));
    if (p->dev_stats) PIPE_CUDA(cudaMemsetAsync(p->dev_stats, 0, 4 * sizeof(int32_t), S(stream)));
    // the ring entry is read by the copy above: it is reused only after step
    // MOE_CACHE_RING - 1's read-back, which the stream orders after it
    return MOE_OK;
}

moe_status moe_cache_step(const moe_dims* dims, const moe_layer_args* args, const moe_layer_outputs* O,
                          moe_cache_pipe* p, const void* const* host_w_gate, const void* const* host_w_up,
                          const void* const* host_w_down, void* const* dev_w_gate, void* const* dev_w_up,
                          void* const* dev_w_down, void* ws, size_t ws_bytes, void* stream, void* stage_stream) {
    size_t need = 0;
    PIPE_TRY(moe_workspace_size(dims, &need));
    if (!pipe_ok(dims, p) || !args || !O || !host_w_gate || !host_w_up || !host_w_down || !dev_w_gate ||
        !dev_w_up || !dev_w_down || !O->topk_idx)
        return MOE_ERR_INVALID_ARG;
    const Homes h{host_w_gate, host_w_up, host_w_down, dev_w_gate, dev_w_up, dev_w_down};
    cudaStream_t s = S(stream);

    // (1) copies that completed; earlier steps' read-backs that are ready
    poll_flights(p);
    PIPE_TRY(consume_ready(dims, p, h, stage_stream));
    // the ring entry of this step must be free: the step MOE_CACHE_RING back
    // has to be consumed (only waits if the host ran far ahead of the GPU)
    while (p->consumed <= p->step - MOE_CACHE_RING) {
        PIPE_CUDA(cudaEventSynchronize(E(p->step_events[p->consumed % MOE_CACHE_RING])));
        PIPE_TRY(consume(dims, p, p->consumed, h, stage_stream));
        ++p->consumed;
    }
    uint64_t* ring = p->host_ring + (size_t)(p->step % MOE_CACHE_RING) * 4;
    uint64_t* cache_d = p->dev_masks + 0;
    uint64_t* resident_d = p->dev_masks + 2;
    uint64_t* admit_d = p->dev_masks + 3;
    const uint64_t landed_now = p->landed;  // forms the next resident set (by value)
    moe_layer_args a = *args;
    a.resident = resident_d;
    a.n_resident = 0;

    if (args->policy != MOE_MISS_EXACT) {
        // (3) the layer on the resident set (stall-free miss handling)
        PIPE_TRY(moe_layer_forward(dims, &a, O, ws, ws_bytes, stream));
    } else {
        // (3') EXACT: the misses must be on the device before the expert FFN
        PIPE_TRY(moe_route(dims, a.x, a.w_router, a.router_bias, a.x_pre, a.w_prefetch, a.w_ord, a.theta, a.tau, 0,
                           O->topk_idx, O->topk_gate, O->router_prob, O->delta_hat, O->prefetch_mask, O->delta_star,
                           nullptr, ws, ws_bytes, stream));
        if (!O->fetch_mask) return MOE_ERR_INVALID_ARG;
        PIPE_TRY(moe_select_resident(dims, O->router_prob, O->topk_idx,
                                     a.use_prefetch_mask ? O->prefetch_mask : nullptr, resident_d, MOE_MISS_EXACT,
                                     0.f, O->delta_hat, O->delta_star, O->final_idx, O->final_gate, O->final_kind,
                                     O->fetch_mask, O->counters, ws, ws_bytes, stream));
        PIPE_CUDA(cudaMemcpyAsync(ring + 3, O->fetch_mask, sizeof(uint64_t), cudaMemcpyDeviceToHost, s));
        PIPE_CUDA(cudaStreamSynchronize(s));
        poll_flights(p);
        const uint64_t fetch = ring[3];
        // in flight: the GPU waits for those copies (they land before the layer)
        for (int f = 0; f < MOE_CACHE_FLIGHTS; ++f)
            if (p->flight_mask[f] & fetch) {
                PIPE_CUDA(cudaStreamWaitEvent(s, E(p->copy_events[f]), 0));
                p->in_time_experts += __builtin_popcountll(p->flight_mask[f] & fetch);
            }
        // landed but not yet in this step's resident set (the one-step lag)
        p->in_time_experts += __builtin_popcountll(fetch & p->landed);
        const uint64_t cold = fetch & ~p->landed & ~p->in_flight;
        if (cold) {
            int f = -1;
            for (int i = 0; i < MOE_CACHE_FLIGHTS; ++i)
                if (!p->flight_mask[i]) { f = i; break; }
            if (f < 0) {  // every slot busy: wait for the oldest-queued copies to finish
                PIPE_CUDA(cudaStreamSynchronize(S(stage_stream)));
                poll_flights(p);
                f = 0;
            }
            const int keep_bound = p->max_flight_experts;
            p->max_flight_experts = 0;  // an on-demand copy is never held back
            int used = -1;
            const moe_status st = stage(dims, p, cold, h, stage_stream, &used);
            p->max_flight_experts = keep_bound;
            PIPE_TRY(st);
            if (used >= 0) PIPE_CUDA(cudaStreamWaitEvent(s, E(p->copy_events[used]), 0));
            p->stall_experts += __builtin_popcountll(cold);
            p->stall_steps += 1;
        }
        PIPE_TRY(moe_permute(dims, O->final_idx, O->final_kind, O->expert_offsets, O->perm, O->inv_perm, ws, ws_bytes,
                             stream));
        PIPE_TRY(moe_expert_ffn(dims, a.x, a.table, O->expert_offsets, O->perm, a.keep_frac, O->y_perm, O->y_shared,
                                ws, ws_bytes, stream));
        PIPE_TRY(moe_combine(dims, O->y_perm, O->inv_perm, O->final_gate, O->final_kind,
                             dims->n_shared > 0 ? O->y_shared : nullptr, nullptr, O->out, stream));
    }

    // (4) heat and cache; the next step's resident set = new cache & landed;
    //     the masks (cache, landed, resident, admit) back to the host ring,
    //     consumed by a later step
    uint64_t* rb = p->dev_ring ? p->dev_ring + (size_t)(p->step % MOE_CACHE_RING) * 4 : nullptr;
    PIPE_CUDA(moe::launch_cache_update(O->topk_idx, dims->T * dims->k, dims->N, p->decay, p->capacity, p->dev_heat,
                                       cache_d, admit_d, p->dev_stats, s, landed_now, resident_d, rb));
    moe::note_launches(1);
    if (!rb) {
        ring[1] = landed_now;
        PIPE_CUDA(cudaMemcpyAsync(ring, p->dev_masks, sizeof(uint64_t), cudaMemcpyDeviceToHost, s));
        PIPE_CUDA(cudaMemcpyAsync(ring + 2, p->dev_masks + 2, 2 * sizeof(uint64_t), cudaMemcpyDeviceToHost, s));
    }
    PIPE_CUDA(cudaEventRecord(E(p->step_events[p->step % MOE_CACHE_RING]), s));
    ++p->step;
    return MOE_OK;
}

moe_status moe_cache_drain(const moe_dims* dims, moe_cache_pipe* p, const void* const* host_w_gate,
                           const void* const* host_w_up, const void* const* host_w_down, void* const* dev_w_gate,
                           void* const* dev_w_up, void* const* dev_w_down, void* stage_stream) {
    if (!pipe_ok(dims, p) || !host_w_gate || !host_w_up || !host_w_down || !dev_w_gate || !dev_w_up || !dev_w_down)
        return MOE_ERR_INVALID_ARG;
    const Homes h{host_w_gate, host_w_up, host_w_down, dev_w_gate, dev_w_up, dev_w_down};
    while (p->consumed < p->step) {
        PIPE_CUDA(cudaEventSynchronize(E(p->step_events[p->consumed % MOE_CACHE_RING])));
        PIPE_TRY(consume(dims, p, p->consumed, h, stage_stream));
        ++p->consumed;
    }
    // every member of the last cache lands, whatever the in-flight bound
    const uint64_t last = p->step > 0 ? p->host_ring[(size_t)((p->step - 1) % MOE_CACHE_RING) * 4] : p->landed;
    const int bound = p->max_flight_experts;
    p->max_flight_experts = 0;
    moe_status st = MOE_OK;
    for (int round = 0; round <= MOE_CACHE_FLIGHTS && st == MOE_OK; ++round) {
        if (cudaStreamSynchronize(S(stage_stream)) != cudaSuccess) { st = MOE_ERR_CUDA; break; }
        poll_flights(p);
        if (!(last & ~p->landed & ~p->in_flight)) break;
        int f;
        st = stage(dims, p, last, h, stage_stream, &f);
    }
    p->max_flight_experts = bound;
    if (st != MOE_OK) return st;
    PIPE_CUDA(cudaStreamSynchronize(S(stage_stream)));
    poll_flights(p);
    return MOE_OK;
}

}  // extern "C"
