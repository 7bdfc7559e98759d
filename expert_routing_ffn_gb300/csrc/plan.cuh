// Token permutation of small batches and the FFN work plans, as block-level
// device functions (used by the permute kernels and by the fused routing
// front end of the layer forward).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

// Exclusive block-wide scan of one int per thread (blockDim.x a multiple of
// 32, at most 1024); returns the thread's prefix, *total the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* total) {
    __shared__ int warp_sums[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    __syncthreads();  // warp_sums may still be read by a previous call
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        if (lane < nw) warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + incl - v;
    *total = warp_sums[nw - 1];
    return before;
}

// FFN plan for the GEMV and decode tensor-core paths, built by a whole block
// (every thread must call it; `off` = expert_offsets[0..N] in shared memory).
// Segments: shared experts first (rows = tokens, in groups of rg), then each
// routed expert's permuted rows in groups of rg.  Channels of all segments
// form one list split over G CTAs in ranges of P (a multiple of p_align);
// see Seg in common.cuh.
__device__ __forceinline__ void build_plan(const PlanArgs& a, const int* off) {
    __shared__ int seg_start[kMaxExperts + 9];  // per expert slot: shared s, then routed e
    __shared__ int s_n;
    const int T = a.T, N = a.N, ns = a.n_shared, rg = a.rg, G = a.G;
    const int n_slots = ns + N;
    const int tid = threadIdx.x;
    int cnt = 0;
    if (tid < n_slots) {
        const int rows = tid < ns ? T : off[tid - ns + 1] - off[tid - ns];
        cnt = (rows + rg - 1) / rg;
    }
    int tot;
    const int first = block_exclusive_scan(cnt, &tot);
    if (tid < n_slots) seg_start[tid] = first;
    if (tid == 0) { seg_start[n_slots] = tot; s_n = tot; }
    __syncthreads();
    const int n = s_n;
    PlanHeader h;
    h.G = G; h.rg = rg; h.n_seg = 0; h.total_ch = 0; h.P = 1; h.n_partial_rows = 0; h.n_routed_rows = 0;
    // A plan that does not fit the workspace is published empty (no segment,
    // no channel, no routed row): the FFN kernels then do nothing, and the
    // error word says why, instead of indexing past the tables.
    if (n > a.max_segs) {
        if (tid == 0) { set_error(a.err, MOE_ERR_CAPACITY, n); *a.hdr = h; }
        return;
    }
    if (tid < n_slots) a.seg_first[tid < ns ? N + tid : tid - ns] = seg_start[tid];
    if (tid == 0) a.seg_first[N + ns] = n;
    const int ns_segs = ns > 0 ? seg_start[ns] : 0;  // shared segments come first
    const int total_ch = ns_segs * a.I_shared + (n - ns_segs) * a.I;
    const int al = a.p_align > 1 ? a.p_align : 1;
    const int P = total_ch > 0 ? ((total_ch + G - 1) / G + al - 1) / al * al : al;
    // one thread per segment (in passes of blockDim.x), partial-row bases by scan
    int carry = 0;
    for (int base = 0; base < n; base += blockDim.x) {
        const int i = base + tid;
        Seg S;
        int w = 0;
        if (i < n) {
            // expert slot of segment i: the last slot whose first segment is <= i
            int lo = 0, hi = n_slots - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (seg_start[mid] <= i) lo = mid; else hi = mid - 1;
            }
            const int j = i - seg_start[lo];  // segment index within the slot
            if (lo < ns) {
                S.expert = N + lo; S.row0 = j * rg; S.rows = min(rg, T - j * rg); S.I = a.I_shared;
                S.ch_start = i * a.I_shared;
            } else {
                const int e = lo - ns;
                S.expert = e; S.row0 = off[e] + j * rg; S.rows = min(rg, off[e + 1] - S.row0); S.I = a.I;
                S.ch_start = ns_segs * a.I_shared + (i - ns_segs) * a.I;
            }
            S.c0 = S.ch_start / P;
            S.npieces = (S.ch_start + S.I - 1) / P - S.c0 + 1;
            S.list_off = -1;
            w = S.npieces * S.rows;
        }
        int tw;
        const int pb = block_exclusive_scan(w, &tw);
        if (i < n) {
            S.pbase = carry + pb;
            a.segs[i] = S;
        }
        carry += tw;
    }
    if (tid == 0) {
        if (carry > a.max_partial_rows) {
            set_error(a.err, MOE_ERR_CAPACITY, carry);
            *a.hdr = h;
            return;
        }
        h.n_seg = n; h.total_ch = total_ch; h.P = P; h.n_partial_rows = carry; h.n_routed_rows = off[N];
        *a.hdr = h;
    }
}

// Tensor-core plan (see TcPlan): shared-expert group first, then every
// routed expert with rows, in expert order.  Built by a whole block (every
// thread calls it; N <= blockDim.x): thread e places expert e's segment from
// one scan of (has rows, row tiles) packed as count + (tiles << 8).
__device__ __forceinline__ void build_tc_plan(const PlanArgs& a, const int* off) {
    TcPlan& P = *a.tc_plan;
    const int tid = threadIdx.x;
    const int n1 = a.I / 128, n2 = a.d / 256;
    const bool sh = a.n_shared > 0;
    const int sh_m = sh ? (a.T + 127) / 128 : 0, sh_n1 = sh ? a.n_shared * a.I_shared / 128 : 0;
    const int sh_p = sh ? (a.T + 255) / 256 : 0;
    int rows = 0, m = 0, mp = 0;
    if (tid < a.N) {
        rows = off[tid + 1] - off[tid];
        m = (rows + 127) / 128;
        mp = (rows + 255) / 256;
    }
    int tot, tot_p;
    const int before = block_exclusive_scan((rows > 0 ? 1 : 0) | (m << 8), &tot);
    const int before_p = block_exclusive_scan(mp, &tot_p);
    if (rows > 0) {
        TcSeg& s = P.seg[(sh ? 1 : 0) + (before & 0xff)];
        const int m_prev = before >> 8;
        s.shared = 0; s.expert = tid; s.row0 = off[tid]; s.rows = rows; s.m_tiles = m; s.n1 = n1;
        s.tile1 = sh_m * sh_n1 + m_prev * n1;
        s.tile2 = sh_m * n2 + m_prev * n2;
        s.mbase = sh_m + m_prev;
        s.m_pairs = mp;
        s.tile1p = sh_p * sh_n1 + before_p * n1;
        s.tile2p = sh_p * n2 + before_p * n2;
    }
    if (tid == 0) {
        if (sh) {
            TcSeg& s = P.seg[0];
            s.shared = 1; s.expert = a.N; s.row0 = 0; s.rows = a.T; s.m_tiles = sh_m; s.n1 = sh_n1;
            s.tile1 = 0; s.tile2 = 0; s.mbase = 0;
            s.m_pairs = sh_p; s.tile1p = 0; s.tile2p = 0;
        }
        P.n_mt = sh_m + (tot >> 8);
        P.n_seg = (sh ? 1 : 0) + (tot & 0xff);
        P.n_tiles1 = sh_m * sh_n1 + (tot >> 8) * n1;
        P.n_tiles2 = sh_m * n2 + (tot >> 8) * n2;
        P.n_tiles1p = sh_p * sh_n1 + tot_p * n1;
        P.n_tiles2p = sh_p * n2 + tot_p * n2;
    }
}

// Up to blockDim.x (<= 1024) slots: one block, one thread per slot.  Slots with the same
// expert in a warp are ranked by __match_any_sync; per-warp counts per expert,
// scanned over warps and then over experts, give every slot its position
// (stable in slot order, as in permute_kernel).  The same block then builds
// the FFN plan.
__device__ __forceinline__ void permute_block(const int32_t* __restrict__ final_idx,
                                              const int32_t* __restrict__ final_kind, int n_slots, int N,
                                              int32_t* __restrict__ expert_offsets, int32_t* __restrict__ perm,
                                              int32_t* __restrict__ inv_perm, DevError* __restrict__ err,
                                              const PlanArgs& plan) {
    __shared__ int cnt[32][kMaxExperts];  // per warp and expert: count, then exclusive prefix over warps
    __shared__ int s_off[kMaxExperts + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    for (int i = tid; i < 32 * kMaxExperts; i += blockDim.x) (&cnt[0][0])[i] = 0;
    int key = -1;  // expert of this slot, -1: no GPU-computed expert (LoRE, host, empty, past the end)
    bool host = false;
    if (tid < n_slots) {
        const int x = final_idx[tid];
        const int kd = final_kind[tid];
        if (x >= N) set_error(err, MOE_ERR_DEVICE_INDEX, tid);
        host = kd == MOE_KIND_CPU;
        if (x >= 0 && x < N && (kd == MOE_KIND_COMPUTE || kd == MOE_KIND_FETCH)) key = x;
    }
    __syncthreads();
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (key >= 0 && rank == 0) cnt[warp][key] = __popc(peers);
    __syncthreads();
    int tot = 0;
    if (tid < N) {
        for (int w = 0; w < nw; ++w) {
            const int c = cnt[w][tid];
            cnt[w][tid] = tot;
            tot += c;
        }
    }
    int all;
    const int first = block_exclusive_scan(tid < N ? tot : 0, &all);
    if (tid < N) s_off[tid] = first;
    if (tid == 0) s_off[N] = all;
    __syncthreads();
    if (tid <= N) expert_offsets[tid] = s_off[tid];
    if (tid < n_slots) {
        if (key >= 0) {
            const int pos = s_off[key] + cnt[warp][key] + rank;
            perm[pos] = tid;
            inv_perm[tid] = pos;
        } else if (!host) {  // host slots keep the position moe_select_hetero gave them
            inv_perm[tid] = -1;
        }
    }
    // only the plan of the path moe_expert_ffn will take
    if (plan.tc_plan) {
        build_tc_plan(plan, s_off);
    } else {
        build_plan(plan, s_off);
    }
}

}  // namespace moe
