// Persistent expert cache across decode steps.
//
// ELMoE-3D (CSDN post), expert-axis elasticity: the system counts how often
// the routing function selects each expert ("heat"), keeps the most
// frequently activated top-K experts resident, and refreshes that subset as
// the activation pattern drifts; its practice note decays every heat by a
// factor just below 1 per time step so that recent activity weighs more.
// One decode step here, after the layer ran with resident = *cache:
//   heat[e] <- decay * heat[e] + #{routed slots of this step on e}
//   cache   <- the `capacity` experts of largest heat, lowest index on ties
//   admit   <- new cache & ~old cache (the experts to stage in before the
//              next step), plus hit / slot / admit / evict counters.
// With a resident output (the overlapped cache pipeline, which passes the
// landed mask, the experts whose weights have arrived, by value) it also
// writes resident <- new cache & landed, the set the next step runs on,
// counts hits against the old resident set (what the step actually ran on)
// instead of the old cache, and may write the four masks into a read-back
// entry that the host can read (mapped pinned memory).
// One block of 64 threads (N <= 64): a shared-memory histogram of the routed
// slots, the heat update, then every thread ranks its expert against all
// others and a ballot forms the new cache.
#include "common.cuh"
#include "kernels.h"

namespace moe {

__global__ void __launch_bounds__(64) cache_update_kernel(const int32_t* __restrict__ topk_idx, int n_slots, int N,
                                                          float decay, int capacity, float* __restrict__ heat,
                                                          uint64_t* __restrict__ cache, uint64_t* __restrict__ admit,
                                                          int32_t* __restrict__ stats, uint64_t landed,
                                                          uint64_t* __restrict__ resident,
                                                          uint64_t* __restrict__ readback) {
    __shared__ int cnt[kMaxExperts];
    __shared__ float h[kMaxExperts];
    __shared__ uint32_t bits[2];
    __shared__ int s_hits[2], s_slots[2];
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
    cnt[e] = 0;
    __syncthreads();
    const uint64_t old = *cache;
    const uint64_t ran_on = resident ? *resident : old;  // the set this step's layer used
    for (int i = e; i < n_slots; i += blockDim.x) {
        const int x = topk_idx[i];
        if (x >= 0 && x < N) atomicAdd(&cnt[x], 1);
    }
    __syncthreads();
    // the heat update, as a rounded product then a rounded sum (no fused
    // multiply-add: the same two roundings on every device)
    if (e < N) h[e] = __fadd_rn(__fmul_rn(decay, heat[e]), (float)cnt[e]);
    __syncthreads();
    int rank = 0;
    if (e < N)
        for (int j = 0; j < N; ++j) rank += (h[j] > h[e] || (h[j] == h[e] && j < e)) ? 1 : 0;
    const bool in = e < N && rank < capacity;
    const uint32_t b = __ballot_sync(0xffffffffu, in);
    // hits: routed slots whose expert was in the old cache
    int hit = (e < N && ((ran_on >> e) & 1)) ? cnt[e] : 0, slots = e < N ? cnt[e] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        hit += __shfl_xor_sync(0xffffffffu, hit, o);
        slots += __shfl_xor_sync(0xffffffffu, slots, o);
    }
    if (lane == 0) { bits[warp] = b; s_hits[warp] = hit; s_slots[warp] = slots; }
    __syncthreads();
    if (e < N) heat[e] = h[e];
    if (e == 0) {
        const uint64_t nw = (uint64_t)bits[0] | ((uint64_t)bits[1] << 32);
        *cache = nw;
        if (admit) *admit = nw & ~old;
        if (resident) *resident = nw & landed;
        if (readback) {  // cache, landed, resident, admit: straight into the host's read-back entry
            readback[0] = nw;
            readback[1] = landed;
            readback[2] = nw & landed;
            readback[3] = nw & ~old;
        }
        if (stats) {
            stats[0] += s_hits[0] + s_hits[1];
            stats[1] += s_slots[0] + s_slots[1];
            stats[2] += __popcll(nw & ~old);
            stats[3] += __popcll(old & ~nw);
        }
    }
}

cudaError_t launch_cache_update(const int32_t* topk_idx, int n_slots, int N, float decay, int capacity, float* heat,
                                uint64_t* cache, uint64_t* admit, int32_t* stats, cudaStream_t st, uint64_t landed,
                                uint64_t* resident, uint64_t* readback) {
    cache_update_kernel<<<1, 64, 0, st>>>(topk_idx, n_slots, N, decay, capacity, heat, cache, admit, stats, landed,
                                          resident, readback);
    return cudaGetLastError();
}

}  // namespace moe
