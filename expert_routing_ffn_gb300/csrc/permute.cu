// Stage 3a: token permutation by expert, and the FFN work plan.
//
// The layer's slots (t, s) that compute an expert (kinds COMPUTE and FETCH)
// are grouped by expert into contiguous segments, stable in (t, s) order, so
// that each expert's weights are streamed once for all of its tokens.
#include "common.cuh"
#include "kernels.h"

namespace moe {

__device__ void build_plan(const PlanArgs& a, const int* off);
__device__ void build_tc_plan(const PlanArgs& a, const int* off);

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
        if (tid == 0) {
            // only the plan of the path moe_expert_ffn will take
            if (plan.tc_plan) build_tc_plan(plan, s_offsets);
            else build_plan(plan, s_offsets);
            *ticket = 0;
        }
    }
}

// FFN plan for the GEMV path (one thread, sequential over segments).
// Segments: shared experts first (rows = tokens, in groups of rg), then each
// routed expert's permuted rows in groups of rg.  Channels of all segments
// form one list split evenly over G CTAs; see Seg in common.cuh.
// `off` holds expert_offsets[0..N] (shared memory).
__device__ void build_plan(const PlanArgs& a, const int* off) {
    const int T = a.T, N = a.N, n_shared = a.n_shared, rg = a.rg, G = a.G;
    int n = 0, ch = 0;
    auto add = [&](int expert, int row0, int rows, int Ie) {
        if (n < a.max_segs) {
            Seg s;
            s.expert = expert; s.row0 = row0; s.rows = rows; s.I = Ie; s.ch_start = ch;
            s.c0 = 0; s.npieces = 0; s.pbase = 0; s.list_off = -1;
            a.segs[n] = s;
        }
        ++n;
        ch += Ie;
    };
    for (int s = 0; s < n_shared; ++s) {
        a.seg_first[N + s] = n;
        for (int r = 0; r < T; r += rg) add(N + s, r, min(rg, T - r), a.I_shared);
    }
    for (int e = 0; e < N; ++e) {
        a.seg_first[e] = n;
        const int lo = off[e], hi = off[e + 1];
        for (int r = lo; r < hi; r += rg) add(e, r, min(rg, hi - r), a.I);
    }
    a.seg_first[N + n_shared] = n;
    PlanHeader h;
    h.G = G; h.rg = rg;
    // A plan that does not fit the workspace is published empty (no segment,
    // no channel, no routed row): the FFN kernels then do nothing, and the
    // error word says why, instead of indexing past the tables.
    auto publish_empty = [&](int detail) {
        set_error(a.err, MOE_ERR_CAPACITY, detail);
        h.n_seg = 0; h.total_ch = 0; h.P = 1; h.n_partial_rows = 0; h.n_routed_rows = 0;
        *a.hdr = h;
    };
    if (n > a.max_segs) { publish_empty(n); return; }
    const int al = a.p_align > 1 ? a.p_align : 1;
    const int P = ch > 0 ? ((ch + G - 1) / G + al - 1) / al * al : al;
    int pbase = 0;
    for (int i = 0; i < n; ++i) {
        Seg& s = a.segs[i];
        s.c0 = s.ch_start / P;
        s.npieces = (s.ch_start + s.I - 1) / P - s.c0 + 1;
        s.pbase = pbase;
        pbase += s.npieces * s.rows;
    }
    if (pbase > a.max_partial_rows) { publish_empty(pbase); return; }
    h.n_seg = n; h.total_ch = ch; h.P = P; h.n_partial_rows = pbase;
    h.n_routed_rows = off[N];
    *a.hdr = h;
}

// Tensor-core plan (see TcPlan): shared-expert group first, then every
// routed expert with rows.
__device__ void build_tc_plan(const PlanArgs& a, const int* off) {
    TcPlan& P = *a.tc_plan;
    int n = 0, t1 = 0, t2 = 0;
    const int n2 = a.d / 256;
    auto add = [&](int shared, int expert, int row0, int rows, int n1) {
        TcSeg& s = P.seg[n++];
        s.shared = shared; s.expert = expert; s.row0 = row0; s.rows = rows;
        s.m_tiles = (rows + 127) / 128; s.n1 = n1; s.tile1 = t1; s.tile2 = t2;
        t1 += s.m_tiles * n1;
        t2 += s.m_tiles * n2;
    };
    if (a.n_shared > 0) add(1, a.N, 0, a.T, a.n_shared * a.I_shared / 128);
    for (int e = 0; e < a.N; ++e)
        if (off[e + 1] > off[e]) add(0, e, off[e], off[e + 1] - off[e], a.I / 128);
    P.n_seg = n; P.n_tiles1 = t1; P.n_tiles2 = t2;
}

__global__ void plan_gemv_kernel(PlanArgs a) {
    __shared__ int off[kMaxExperts + 1];
    for (int i = threadIdx.x; i <= a.N; i += blockDim.x) off[i] = __ldcg(&a.expert_offsets[i]);
    __syncthreads();
    if (threadIdx.x == 0) build_plan(a, off);
}

cudaError_t launch_permute(const PermuteArgs& a, const PlanArgs& plan, int* ticket,
                           cudaStream_t st) {
    permute_kernel<<<a.N, 1024, 0, st>>>(a.final_idx, a.final_kind, a.n_slots, a.N,
                                         a.expert_offsets, a.perm, a.inv_perm, a.err, plan, ticket);
    return cudaGetLastError();
}

cudaError_t launch_plan_gemv(const PlanArgs& a, cudaStream_t st) {
    plan_gemv_kernel<<<1, 32, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
