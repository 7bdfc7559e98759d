// Stage 3a: token permutation by expert, and the FFN work plan.
//
// The layer's slots (t, s) that compute an expert (kinds COMPUTE and FETCH)
// are grouped by expert into contiguous segments, stable in (t, s) order, so
// that each expert's weights are streamed once for all of its tokens.
#include "common.cuh"
#include "kernels.h"
#include "plan.cuh"

namespace moe {


// Batches of more than 1024 slots: two launches over chunks of kPermChunk
// slots, one block (one thread per slot) per chunk.
//  1. permute_count_kernel: the chunk's slot count per expert -> counts[c][e].
//  2. permute_scatter_kernel: every block scans the count table (expert
//     offsets, and the slots of earlier chunks per expert), ranks its slots
//     within the chunk (per-warp ranks by __match_any_sync, then earlier warps)
//     and scatters them; the order is stable in slot order, as in
//     permute_block.  Block 0 writes expert_offsets and builds the FFN plan.
// LORE = true groups the LoRE slots instead (moe_lore's grouped path; no plan).
template <bool LORE>
__device__ __forceinline__ int permute_key(const int32_t* __restrict__ final_idx,
                                           const int32_t* __restrict__ final_kind, int i, int n_slots, int N,
                                           DevError* __restrict__ err) {
    if (i >= n_slots) return -1;
    const int x = final_idx[i];
    const int kd = final_kind[i];
    const bool lore = kd == MOE_KIND_LORE;
    if (x >= N && (!LORE || lore)) { if (err) set_error(err, MOE_ERR_DEVICE_INDEX, i); return -1; }
    const bool mine = LORE ? lore : (kd == MOE_KIND_COMPUTE || kd == MOE_KIND_FETCH);
    return (x >= 0 && x < N && mine) ? x : -1;
}

// per warp and expert: the warp's slot count; returns this slot's rank among
// the warp's slots of the same expert
__device__ __forceinline__ int permute_warp_counts(int key, int (*cnt)[kMaxExperts]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && __popc(peers & ((1u << lane) - 1u)) == 0) cnt[warp][key] = __popc(peers);
    return __popc(peers & ((1u << lane) - 1u));
}

template <bool LORE>
__global__ void __launch_bounds__(kPermChunk) permute_count_kernel(const int32_t* __restrict__ final_idx,
                                                                   const int32_t* __restrict__ final_kind,
                                                                   int n_slots, int N,
                                                                   int32_t* __restrict__ counts,
                                                                   DevError* __restrict__ err) {
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
    __shared__ int cnt[kPermChunk / 32][kMaxExperts];
    const int tid = threadIdx.x, nw = blockDim.x >> 5;
    for (int i = tid; i < nw * kMaxExperts; i += blockDim.x) (&cnt[0][0])[i] = 0;
    __syncthreads();
    const int key = permute_key<LORE>(final_idx, final_kind, blockIdx.x * kPermChunk + tid, n_slots, N, err);
    (void)permute_warp_counts(key, cnt);
    __syncthreads();
    if (tid < N) {
        int tot = 0;
        for (int w = 0; w < nw; ++w) tot += cnt[w][tid];
        counts[(size_t)blockIdx.x * kMaxExperts + tid] = tot;
    }
    grid_dep_launch();
}

template <bool LORE>
__global__ void __launch_bounds__(kPermChunk) permute_scatter_kernel(const int32_t* __restrict__ final_idx,
                                                                     const int32_t* __restrict__ final_kind,
                                                                     int n_slots, int N,
                                                                     const int32_t* __restrict__ counts,
                                                                     int32_t* __restrict__ expert_offsets,
                                                                     int32_t* __restrict__ perm,
                                                                     int32_t* __restrict__ inv_perm,
                                                                     PlanArgs plan) {
    __shared__ int cnt[kPermChunk / 32][kMaxExperts];  // per warp and expert, then exclusive over warps
    __shared__ int base[kMaxExperts];                    // first position of this chunk's slots per expert
    __shared__ int s_off[kMaxExperts + 1];
    const int c = blockIdx.x, n_chunks = gridDim.x;
    const int tid = threadIdx.x, warp = tid >> 5, nw = blockDim.x >> 5;
    for (int i = tid; i < nw * kMaxExperts; i += blockDim.x) (&cnt[0][0])[i] = 0;
    const int slot = c * kPermChunk + tid;
    // final_idx / final_kind come from the previous kernels (the count
    // kernel reported bad indices already)
    grid_dep_wait();
    const int key = permute_key<LORE>(final_idx, final_kind, slot, n_slots, N, nullptr);
    __syncthreads();
    const int rank = permute_warp_counts(key, cnt);
    // expert totals and this chunk's start per expert, from the count table
    int before = 0, tot = 0;
    if (tid < N) {
        for (int q = 0; q < n_chunks; ++q) {
            const int v = __ldcg(counts + (size_t)q * kMaxExperts + tid);
            if (q < c) before += v;
            tot += v;
        }
    }
    int all;
    const int first = block_exclusive_scan(tid < N ? tot : 0, &all);  // syncs: cnt complete after it
    if (tid < N) { s_off[tid] = first; base[tid] = first + before; }
    if (tid == 0) s_off[N] = all;
    if (tid < N) {
        int run = 0;
        for (int w = 0; w < nw; ++w) {
            const int v = cnt[w][tid];
            cnt[w][tid] = run;
            run += v;
        }
    }
    __syncthreads();
    if (slot < n_slots) {
        if (key >= 0) {
            const int pos = base[key] + cnt[warp][key] + rank;
            perm[pos] = slot;
            inv_perm[slot] = pos;
        } else if (LORE || final_kind[slot] != MOE_KIND_CPU) {
            inv_perm[slot] = -1;  // host slots keep the position moe_select_hetero gave them
        }
    }
    if (c == 0) {
        if (tid <= N) expert_offsets[tid] = s_off[tid];
        if (LORE) return;
        // only the plan of the path moe_expert_ffn will take
        if (plan.tc_plan) {
            build_tc_plan(plan, s_off);
        } else {
            build_plan(plan, s_off);
        }
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

cudaError_t launch_permute(const PermuteArgs& a, const PlanArgs& plan, int32_t* counts,
                           cudaStream_t st) {
    if (a.n_slots <= 1024) {
        const int threads = a.n_slots <= 256 ? 256 : 1024;
        permute_small_kernel<<<1, threads, 0, st>>>(a.final_idx, a.final_kind, a.n_slots, a.N,
                                                   a.expert_offsets, a.perm, a.inv_perm, a.err, plan);
        return cudaGetLastError();
    }
    const int n_chunks = (a.n_slots + kPermChunk - 1) / kPermChunk;
    cudaError_t e = launch_pdl(permute_count_kernel<false>, dim3(n_chunks), dim3(kPermChunk), 0, st, a.final_idx,
                               a.final_kind, a.n_slots, a.N, counts, a.err);
    if (e != cudaSuccess) return e;
    return launch_pdl(permute_scatter_kernel<false>, dim3(n_chunks), dim3(kPermChunk), 0, st, a.final_idx,
                      a.final_kind, a.n_slots, a.N, (const int32_t*)counts, a.expert_offsets, a.perm,
                      a.inv_perm, plan);
}

cudaError_t launch_group_lore(const PermuteArgs& a, int32_t* counts, cudaStream_t st) {
    const int n_chunks = (a.n_slots + kPermChunk - 1) / kPermChunk;
    cudaError_t e = launch_pdl(permute_count_kernel<true>, dim3(n_chunks), dim3(kPermChunk), 0, st, a.final_idx,
                               a.final_kind, a.n_slots, a.N, counts, a.err);
    if (e != cudaSuccess) return e;
    PlanArgs none;
    none.tc_plan = nullptr;
    return launch_pdl(permute_scatter_kernel<true>, dim3(n_chunks), dim3(kPermChunk), 0, st, a.final_idx,
                      a.final_kind, a.n_slots, a.N, (const int32_t*)counts, a.expert_offsets, a.perm,
                      a.inv_perm, none);
}

cudaError_t launch_plan_gemv(const PlanArgs& a, cudaStream_t st) {
    plan_gemv_kernel<<<1, 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
