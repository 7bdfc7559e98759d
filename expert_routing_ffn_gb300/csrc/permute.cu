// Stage 3a: token permutation by expert, and the FFN work plan.
//
// The layer's slots (t, s) that compute an expert (kinds COMPUTE and FETCH)
// are grouped by expert into contiguous segments, stable in (t, s) order, so
// that each expert's weights are streamed once for all of its tokens.
#include "common.cuh"
#include "kernels.h"
#include "plan.cuh"

namespace moe {


// One block per expert e.  Pass 1 counts the slots routed to experts below e
// (the segment offset) and to e; pass 2 walks the slots in order and
// scatters e's slots with a block-wide prefix over 1024-slot chunks.
// Block 0 also marks LoRE / empty slots with inv_perm = -1.
// The last block to finish (arrival counter `ticket`, left at 0 afterwards)
// also builds the FFN plan from the complete expert_offsets.
__global__ void __launch_bounds__(1024) permute_kernel(const int32_t* __restrict__ final_idx,
                                                       const int32_t* __restrict__ final_kind,
                                                       int n_slots, int N,
                                                       int32_t* __restrict__ expert_offsets,
                                                       int32_t* __restrict__ perm,
                                                       int32_t* __restrict__ inv_perm,
                                                       DevError* __restrict__ err, PlanArgs plan,
                                                       int* __restrict__ ticket) {
    __shared__ int red_less[32], red_eq[32];
    __shared__ int warp_pref[32];
    __shared__ int s_off;
    __shared__ int s_last;
    __shared__ int s_offsets[kMaxExperts + 1];
    const int e = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    int less = 0, eq = 0;
    for (int i = tid; i < n_slots; i += blockDim.x) {
        const int x = final_idx[i];
        const bool valid = x >= 0 && final_kind[i] != MOE_KIND_LORE;
        if (x >= N) { if (e == 0) set_error(err, MOE_ERR_DEVICE_INDEX, i); continue; }
        less += (valid && x < e) ? 1 : 0;
        eq += (valid && x == e) ? 1 : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        less += __shfl_xor_sync(0xffffffffu, less, o);
        eq += __shfl_xor_sync(0xffffffffu, eq, o);
    }
    if (lane == 0) { red_less[warp] = less; red_eq[warp] = eq; }
    __syncthreads();
    if (tid == 0) {
        int L = 0, E = 0;
        for (int w = 0; w < nw; ++w) { L += red_less[w]; E += red_eq[w]; }
        s_off = L;
        expert_offsets[e] = L;
        if (e == N - 1) expert_offsets[N] = L + E;
    }
    __syncthreads();
    int running = s_off;
    for (int base = 0; base < n_slots; base += blockDim.x) {
        const int i = base + tid;
        bool mine = false, valid = false;
        if (i < n_slots) {
            const int x = final_idx[i];
            valid = x >= 0 && x < N && final_kind[i] != MOE_KIND_LORE;
            mine = valid && x == e;
            if (e == 0 && !valid) inv_perm[i] = -1;
        }
        const uint32_t b = __ballot_sync(0xffffffffu, mine);
        if (lane == 0) warp_pref[warp] = __popc(b);
        __syncthreads();
        int before = 0, total = 0;
        for (int w = 0; w < nw; ++w) {
            const int c = warp_pref[w];
            if (w < warp) before += c;
            total += c;
        }
        if (mine) {
            const int pos = running + before + __popc(b & ((1u << lane) - 1u));
            perm[pos] = i;
            inv_perm[i] = pos;
        }
        running += total;
        __syncthreads();
    }
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(ticket, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int i = tid; i <= N; i += blockDim.x) s_offsets[i] = __ldcg(&expert_offsets[i]);
        __syncthreads();
        // only the plan of the path moe_expert_ffn will take
        if (plan.tc_plan) {
            if (tid == 0) build_tc_plan(plan, s_offsets);
        } else {
            build_plan(plan, s_offsets);
        }
        if (tid == 0) *ticket = 0;
    }
}

__global__ void __launch_bounds__(1024) permute_small_kernel(const int32_t* __restrict__ final_idx,
                                                             const int32_t* __restrict__ final_kind,
                                                             int n_slots, int N,
                                                             int32_t* __restrict__ expert_offsets,
                                                             int32_t* __restrict__ perm,
                                                             int32_t* __restrict__ inv_perm,
                                                             DevError* __restrict__ err, PlanArgs plan) {
    permute_block(final_idx, final_kind, n_slots, N, expert_offsets, perm, inv_perm, err, plan);
}

__global__ void __launch_bounds__(256) plan_gemv_kernel(PlanArgs a) {
    __shared__ int off[kMaxExperts + 1];
    for (int i = threadIdx.x; i <= a.N; i += blockDim.x) off[i] = __ldcg(&a.expert_offsets[i]);
    __syncthreads();
    build_plan(a, off);
}

cudaError_t launch_permute(const PermuteArgs& a, const PlanArgs& plan, int* ticket,
                           cudaStream_t st) {
    if (a.n_slots <= 1024) {
        const int threads = a.n_slots <= 256 ? 256 : 1024;
        permute_small_kernel<<<1, threads, 0, st>>>(a.final_idx, a.final_kind, a.n_slots, a.N,
                                                   a.expert_offsets, a.perm, a.inv_perm, a.err, plan);
        return cudaGetLastError();
    }
    permute_kernel<<<a.N, 1024, 0, st>>>(a.final_idx, a.final_kind, a.n_slots, a.N,
                                         a.expert_offsets, a.perm, a.inv_perm, a.err, plan, ticket);
    return cudaGetLastError();
}

cudaError_t launch_plan_gemv(const PlanArgs& a, cudaStream_t st) {
    plan_gemv_kernel<<<1, 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
