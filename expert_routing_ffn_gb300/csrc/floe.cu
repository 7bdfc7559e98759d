// FloE contextual sparsity for routed experts (FloE: On-the-Fly MoE Inference
// on Memory-constrained GPU, method §1: a^S(x) = (SiLU(x W_gate) (.)
// S_t(x W_up)) W_down, the mask S_t keeping the channels with the largest
// |x W_up|; §3: gate and down read only for the kept channels, stored
// channel-contiguous).
//
// Decode path, per call:
//   GEMV, up-only pass  u[pos, i] = x_t . W_up[e][i, :] for every routed row
//                       (dense up projection, every channel; the GEMV kernel
//                       with segments marked kUpOnly)
//   floe_select_kernel  per row: the m channels with the largest |u|
//                       (lowest channel index among equal values) as a bitset
//   floe_union_kernel   per expert: the union of its rows' channel sets as an
//                       ascending channel list (each listed gate/down row is
//                       then read once for all of the expert's rows)
//   floe_plan_kernel    the GEMV plan over the union lists (shared experts
//                       stay dense)
// followed by the GEMV kernel in its sparse mode and the partial reduction.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// Plan of the first FloE pass: every routed expert's rows in groups of 2
// over all I channels, up projection only (no partial outputs).
__global__ void floe_up_plan_kernel(PlanArgs a) {
    __shared__ int off[kMaxExperts + 1];
    for (int i = threadIdx.x; i <= a.N; i += blockDim.x) off[i] = a.expert_offsets[i];
    __syncthreads();
    if (threadIdx.x != 0) return;
    int n = 0, ch = 0;
    for (int e = 0; e < a.N; ++e)
        for (int r = off[e]; r < off[e + 1]; r += 2) {
            if (n < a.max_segs) {
                Seg s;
                s.expert = e; s.row0 = r; s.rows = min(2, off[e + 1] - r); s.I = a.I; s.ch_start = ch;
                s.c0 = 0; s.npieces = 0; s.pbase = 0; s.list_off = kUpOnly;
                a.segs[n] = s;
            }
            ++n;
            ch += a.I;
        }
    PlanHeader h;
    h.G = a.G; h.rg = a.rg; h.n_partial_rows = 0; h.n_routed_rows = off[a.N];
    if (n > a.max_segs) {
        set_error(a.err, MOE_ERR_CAPACITY, n);
        n = 0; ch = 0;
    }
    h.n_seg = n; h.total_ch = ch; h.P = ch > 0 ? (ch + a.G - 1) / a.G : 1;
    *a.hdr = h;
}

// One block per routed row: the m largest |u| (ties: lowest channel index).
// Radix select over the bit patterns of |u| (order-preserving for
// non-negative floats), 8 bits per pass, then a block scan ranks the
// channels equal to the threshold by index.
__global__ void __launch_bounds__(1024) floe_select_kernel(const float* __restrict__ u,
                                                           const int32_t* __restrict__ expert_offsets,
                                                           int N, int I, int m, int words,
                                                           uint32_t* __restrict__ kept) {
    extern __shared__ __align__(16) uint32_t keys[];  // [I] then bitset [words]
    uint32_t* bits = keys + I;
    __shared__ int hist[256];
    __shared__ uint32_t s_prefix;
    __shared__ int s_remaining;
    __shared__ int warp_tot[32];
    const int pos = blockIdx.x;
    if (pos >= expert_offsets[N]) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // |u| as ordered keys: 16-byte loads, all in flight at once (the row was
    // just written by the up pass and sits in L2)
    const float* ur = u + (size_t)pos * I;
    const int I4 = reinterpret_cast<uintptr_t>(ur) % 16 == 0 ? I / 4 : 0;
#pragma unroll 4
    for (int i = tid; i < I4; i += blockDim.x) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(ur) + i);
        reinterpret_cast<uint4*>(keys)[i] = make_uint4(__float_as_uint(fabsf(v.x)), __float_as_uint(fabsf(v.y)),
                                                       __float_as_uint(fabsf(v.z)), __float_as_uint(fabsf(v.w)));
    }
    for (int i = 4 * I4 + tid; i < I; i += blockDim.x) keys[i] = __float_as_uint(fabsf(__ldcg(ur + i)));
    for (int w = tid; w < words; w += blockDim.x) bits[w] = 0u;
    if (tid == 0) { s_prefix = 0u; s_remaining = m; }
    uint32_t mask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        // one shared-memory atomic per key in the current prefix (grouping
        // equal bins of a warp with a match first measured slower: 20.4
        // against 14.8 us for a 14336-channel row)
        for (int base = 0; base < I; base += blockDim.x) {
            const int i = base + tid;
            if (i < I && (keys[i] & mask) == prefix) atomicAdd(&hist[(keys[i] >> shift) & 255u], 1);
        }
        __syncthreads();
        if (warp == 0) {
            // the first bin, in descending order, at which the running count
            // reaches the number still to keep: lane L holds bins 255 - 8L ..
            // 248 - 8L, an exclusive scan over lanes, and the one lane whose
            // span holds the crossing walks its eight bins
            int v[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) { v[j] = hist[255 - (8 * lane + j)]; sum += v[j]; }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            const int rem = s_remaining;
            int cum = incl - sum;
            if (cum < rem && rem <= incl) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (cum + v[j] >= rem) {
                        s_prefix = prefix | ((uint32_t)(255 - (8 * lane + j)) << shift);
                        s_remaining = rem - cum;
                        break;
                    }
                    cum += v[j];
                }
            }
        }
        mask |= 255u << shift;
        __syncthreads();
    }
    const uint32_t thr = s_prefix;
    const int need_eq = s_remaining;  // channels equal to thr that are kept
    // rank the channels equal to thr by index: contiguous chunks per thread
    const int per = (I + blockDim.x - 1) / blockDim.x;
    const int lo = tid * per, hi = min(I, lo + per);
    int n_eq = 0;
    for (int i = lo; i < hi; ++i) n_eq += keys[i] == thr ? 1 : 0;
    int incl = n_eq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = incl - n_eq;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    for (int i = lo; i < hi; ++i) {
        bool keep = keys[i] > thr;
        if (keys[i] == thr) { keep = before < need_eq; ++before; }
        if (keep) atomicOr(&bits[i >> 5], 1u << (i & 31));
    }
    __syncthreads();
    for (int w = tid; w < words; w += blockDim.x) kept[(size_t)pos * words + w] = bits[w];
}

// One block per expert: OR of its rows' bitsets, compacted to an ascending
// channel list; count[e] = its length.
__global__ void __launch_bounds__(512) floe_union_kernel(const uint32_t* __restrict__ kept,
                                                         const int32_t* __restrict__ expert_offsets,
                                                         int I, int words, int32_t* __restrict__ list,
                                                         int32_t* __restrict__ count) {
    __shared__ int warp_tot[16];
    const int e = blockIdx.x;
    const int a = expert_offsets[e], b = expert_offsets[e + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // each thread owns a contiguous run of words
    const int per = (words + blockDim.x - 1) / blockDim.x;
    const int w0 = tid * per, w1 = min(words, w0 + per);
    int n = 0;
    for (int w = w0; w < w1; ++w) {
        uint32_t v = 0u;
        for (int r = a; r < b; ++r) v |= kept[(size_t)r * words + w];
        n += __popc(v);
    }
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = incl - n;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    int32_t* out = list + (size_t)e * I;
    for (int w = w0; w < w1; ++w) {
        uint32_t v = 0u;
        for (int r = a; r < b; ++r) v |= kept[(size_t)r * words + w];
        while (v) {
            const int bit = __ffs(v) - 1;
            out[base++] = w * 32 + bit;
            v &= v - 1;
        }
    }
    if (tid == blockDim.x - 1) count[e] = (a == b) ? 0 : base;
}

// The GEMV plan over union lists: shared experts dense, then each routed
// expert's rows in groups of rg over its count[e] listed channels.
__global__ void floe_plan_kernel(PlanArgs a, const int32_t* __restrict__ count) {
    __shared__ int off[kMaxExperts + 1];
    __shared__ int cnt[kMaxExperts];
    for (int i = threadIdx.x; i <= a.N; i += blockDim.x) off[i] = a.expert_offsets[i];
    for (int i = threadIdx.x; i < a.N; i += blockDim.x) cnt[i] = count[i];
    __syncthreads();
    if (threadIdx.x != 0) return;
    int n = 0, ch = 0;
    auto add = [&](int expert, int row0, int rows, int Ie, int list_off) {
        if (n < a.max_segs) {
            Seg s;
            s.expert = expert; s.row0 = row0; s.rows = rows; s.I = Ie; s.ch_start = ch;
            s.c0 = 0; s.npieces = 0; s.pbase = 0; s.list_off = list_off;
            a.segs[n] = s;
        }
        ++n;
        ch += Ie;
    };
    for (int s = 0; s < a.n_shared; ++s) {
        a.seg_first[a.N + s] = n;
        for (int r = 0; r < a.T; r += a.rg) add(a.N + s, r, min(a.rg, a.T - r), a.I_shared, -1);
    }
    for (int e = 0; e < a.N; ++e) {
        a.seg_first[e] = n;
        for (int r = off[e]; r < off[e + 1]; r += a.rg)
            add(e, r, min(a.rg, off[e + 1] - r), cnt[e], e * a.I);
    }
    a.seg_first[a.N + a.n_shared] = n;
    PlanHeader h;
    h.G = a.G; h.rg = a.rg;
    if (n > a.max_segs) {
        set_error(a.err, MOE_ERR_CAPACITY, n);
        h.n_seg = 0; h.total_ch = 0; h.P = 1; h.n_partial_rows = 0; h.n_routed_rows = 0;
        *a.hdr = h;
        return;
    }
    const int P = ch > 0 ? (ch + a.G - 1) / a.G : 1;
    int pbase = 0;
    for (int i = 0; i < n; ++i) {
        Seg& s = a.segs[i];
        s.c0 = s.ch_start / P;
        s.npieces = s.I > 0 ? (s.ch_start + s.I - 1) / P - s.c0 + 1 : 0;
        s.pbase = pbase;
        pbase += s.npieces * s.rows;
    }
    if (pbase > a.max_partial_rows) {
        set_error(a.err, MOE_ERR_CAPACITY, pbase);
        h.n_seg = 0; h.total_ch = 0; h.P = 1; h.n_partial_rows = 0; h.n_routed_rows = 0;
        *a.hdr = h;
        return;
    }
    h.n_seg = n; h.total_ch = ch; h.P = P; h.n_partial_rows = pbase; h.n_routed_rows = off[a.N];
    *a.hdr = h;
}

cudaError_t launch_floe_prepare(const FloeArgs& f, const PlanArgs& plan, const GemvParams& gp, int G,
                                cudaStream_t st) {
    cudaError_t e;
    if (f.tc_nt > 0) {
        // up pass on the decode tensor cores: the routed rows in segments of
        // tc_nt, 16-aligned channel ranges, U written to u
        PlanArgs pu = plan;
        pu.rg = f.tc_nt; pu.G = f.tc_grid; pu.p_align = 16; pu.n_shared = 0;
        e = launch_plan_gemv(pu, st);
        if (e != cudaSuccess) return e;
        TcdLaunch t;
        t.x = f.x; t.perm = f.perm; t.expert_offsets = f.expert_offsets; t.table = f.table;
        t.hdr = plan.hdr; t.segs = plan.segs; t.x_perm = f.x_perm; t.partial = nullptr;
        t.T = f.T; t.d = f.d; t.N = f.N; t.k = f.topk; t.rows_cap = f.rows_cap; t.nt = f.tc_nt;
        t.grid = f.tc_grid; t.u_out = f.u; t.I = f.I; t.err = plan.err; t.prefetch_shared = 0;
        e = launch_tcd_ffn(t, st);
    } else {
        floe_up_plan_kernel<<<1, 64, 0, st>>>(plan);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        GemvParams up = gp;
        up.up_pass = 1;
        up.prefetch_shared = 0;
        up.NS = gemv_stages(f.d, true);  // the up pass's stages hold 2 x 3 rows
        e = launch_gemv(up, G, true, st, true);
    }
    if (e != cudaSuccess) return e;
    const size_t sel_smem = ((size_t)f.I + f.words) * sizeof(uint32_t);
    e = allow_max_smem(floe_select_kernel);
    if (e != cudaSuccess) return e;
    floe_select_kernel<<<f.rows_cap, 1024, sel_smem, st>>>(f.u, f.expert_offsets, f.N, f.I, f.m,
                                                           f.words, f.kept);
    e = note_launch(reinterpret_cast<const void*>(floe_select_kernel), 1024, sel_smem, cudaGetLastError());
    if (e != cudaSuccess) return e;
    floe_union_kernel<<<f.N, 512, 0, st>>>(f.kept, f.expert_offsets, f.I, f.words, f.list, f.count);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    floe_plan_kernel<<<1, 64, 0, st>>>(plan, f.count);
    return cudaGetLastError();
}

}  // namespace moe
