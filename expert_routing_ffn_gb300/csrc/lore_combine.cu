// Stages 4 and 5: the SPICE LoRE surrogate residual and the combine.
//
// SPICE write-up, LoRE section: a missing expert e is approximated by
// y_shared + B_e A_e h with A_e [r, d], B_e [d, r], r << d; the shared part
// is added once per token by the combine, scaled by the LoRE slots' gates.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// z[t, s, :] = g_s * A_e x_t for a LoRE slot (t, s) (zero for other slots):
// one block per slot, its warps over the r rank rows, lanes over d.
template <typename W>
__global__ void __launch_bounds__(256) lore_z_kernel(const W* __restrict__ x,
                                                     const int32_t* __restrict__ final_idx,
                                                     const int32_t* __restrict__ final_kind,
                                                     const float* __restrict__ final_gate,
                                                     const W* __restrict__ A, int d, int k, int r,
                                                     int N, float* __restrict__ z,
                                                     DevError* __restrict__ err) {
    constexpr int V = Vec<W>::n;
    const int slot = blockIdx.x;
    const int t = slot / k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int q_begin = 0, q_end = r;  // rank rows q = warp, warp + nw, ...
    const int e = final_idx[slot];
    if (final_kind[slot] != MOE_KIND_LORE || e < 0 || e >= N) {
        if (final_kind[slot] == MOE_KIND_LORE && err && tid == 0) set_error(err, MOE_ERR_DEVICE_INDEX, slot);
        for (int q = q_begin + tid; q < q_end; q += blockDim.x) z[(size_t)slot * r + q] = 0.f;
        return;
    }
    const float g = final_gate[slot];
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    const int nchunk = d / V;
    for (int q = q_begin + warp; q < q_end; q += nw) {
        const uint4* arow = reinterpret_cast<const uint4*>(A + ((size_t)e * r + q) * d);
        float acc = 0.f;
        for (int c = lane; c < nchunk; c += 32) {
            float av[V], xv[V];
            unpack16(arow[c], av, (W*)nullptr);
            unpack16(xr[c], xv, (W*)nullptr);
#pragma unroll
            for (int j = 0; j < V; ++j) acc = fmaf(av[j], xv[j], acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) z[(size_t)slot * r + q] = g * acc;
    }
}

// y_lore[t, j] = sum over LoRE slots s of sum_q B_e[j, q] z[t, s, q]:
// blocks over (token, 256 output columns), one column per thread.
template <typename W>
__global__ void __launch_bounds__(256) lore_b_kernel(const int32_t* __restrict__ final_idx,
                                                     const int32_t* __restrict__ final_kind,
                                                     const W* __restrict__ B, int d, int k, int r,
                                                     int N, const float* __restrict__ z,
                                                     float* __restrict__ y_lore) {
    const int t = blockIdx.x;
    const int j = blockIdx.y * blockDim.x + threadIdx.x;
    __shared__ int s_e[kMaxTopK];
    __shared__ float s_z[kMaxTopK * 64];
    __shared__ int s_n;
    if (threadIdx.x < 32) {  // one lane per slot, LoRE slots compacted in slot order
        const int s = threadIdx.x;
        bool is_lore = false;
        if (s < k) {
            const size_t sl = (size_t)t * k + s;
            const int e = final_idx[sl];
            is_lore = final_kind[sl] == MOE_KIND_LORE && e >= 0 && e < N;
        }
        const uint32_t b = __ballot_sync(0xffffffffu, is_lore);
        if (is_lore) s_e[__popc(b & ((1u << s) - 1u))] = s;
        if (s == 0) s_n = __popc(b);
    }
    __syncthreads();
    const int n = s_n;
    for (int i = threadIdx.x; i < n * r; i += blockDim.x)
        s_z[i] = z[((size_t)t * k + s_e[i / r]) * r + (i % r)];
    __syncthreads();
    if (j >= d) return;
    float acc = 0.f;
    for (int i = 0; i < n; ++i) {
        const int e = final_idx[(size_t)t * k + s_e[i]];
        const W* brow = B + ((size_t)e * d + j) * r;
        const float* zz = s_z + i * r;
        if ((r * (int)sizeof(W)) % 16 == 0) {
            // 16-byte loads of the rank row B_e[j, :]
            for (int q = 0; q < r; q += Vec<W>::n) {
                float bv[Vec<W>::n];
                unpack16(*reinterpret_cast<const uint4*>(brow + q), bv, (W*)nullptr);
#pragma unroll
                for (int u = 0; u < Vec<W>::n; ++u) acc = fmaf(bv[u], zz[q + u], acc);
            }
        } else {
            for (int q = 0; q < r; ++q) acc = fmaf(to_f32(brow[q]), zz[q], acc);
        }
    }
    y_lore[(size_t)t * d + j] = acc;
}

// out[t] = y_shared[t] (1 + sum of LoRE gates) + sum_s g_s y_perm[inv_perm[t,s]]
//        + y_lore[t]; slots in order.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y_perm,
                                                      const int32_t* __restrict__ inv_perm,
                                                      const float* __restrict__ final_gate,
                                                      const int32_t* __restrict__ final_kind,
                                                      const float* __restrict__ y_shared,
                                                      const float* __restrict__ y_lore, int d,
                                                      int k, float* __restrict__ out) {
    const int t = blockIdx.x;
    const int q = blockIdx.y * blockDim.x + threadIdx.x;  // float4 column group
    __shared__ int s_pos[kMaxTopK], s_kind[kMaxTopK];
    __shared__ float s_g[kMaxTopK];
    __shared__ float s_lg;
    if (threadIdx.x < k) {  // one thread per slot
        const size_t sl = (size_t)t * k + threadIdx.x;
        s_pos[threadIdx.x] = inv_perm[sl];
        s_g[threadIdx.x] = final_gate[sl];
        s_kind[threadIdx.x] = final_kind[sl];
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // the LoRE gates summed in slot order
        float lg = 0.f;
        for (int s = 0; s < k; ++s)
            if (s_kind[s] == MOE_KIND_LORE) lg += s_g[s];
        s_lg = lg;
    }
    __syncthreads();
    const float sh_scale = 1.f + s_lg;
    if (q < d / 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (y_shared) {
            const float4 v = reinterpret_cast<const float4*>(y_shared + (size_t)t * d)[q];
            acc.x = v.x * sh_scale; acc.y = v.y * sh_scale; acc.z = v.z * sh_scale; acc.w = v.w * sh_scale;
        }
        for (int s = 0; s < k; ++s) {
            const int pos = s_pos[s];
            if (pos < 0) continue;
            const float g = s_g[s];
            const float4 v = reinterpret_cast<const float4*>(y_perm + (size_t)pos * d)[q];
            acc.x = fmaf(g, v.x, acc.x); acc.y = fmaf(g, v.y, acc.y);
            acc.z = fmaf(g, v.z, acc.z); acc.w = fmaf(g, v.w, acc.w);
        }
        if (y_lore) {
            const float4 v = reinterpret_cast<const float4*>(y_lore + (size_t)t * d)[q];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        reinterpret_cast<float4*>(out + (size_t)t * d)[q] = acc;
    }
}

// moe_layer_forward's tail when the expert FFN left per-CTA partial rows
// (GEMV and decode tensor-core paths).  Block = token t x 128 columns of d
// (lane = 4 columns).  A "unit" is one segment row feeding the token: the
// y_perm row of a computed slot, or one shared expert's row.  Warp 0 reads
// the slots; then the last warp forms the LoRE term (z, then B rows times z)
// while the others sum the units:
//  - not DIRECT (GEMV partials, up to eight runs a unit): warp 0 also looks up
//    the units; warps 0..nw-2 sum all units' runs into dynamic shared memory
//    ((k + n_shared) * kSumChunks * 32 float4), then warp s < k adds up slot
//    s's runs and warp kMaxTopK the shared experts';
//  - DIRECT (decode tensor-core partials, a few pieces a segment): warp s < k
//    looks up and sums slot s's unit, warp nw-2 the shared experts'
//    (partial_unit_sum).
// Warp 0 then combines in slot order.  Every sum runs in the order of the
// separate kernels (gemv_reduce_kernel, lore_b_kernel, combine_kernel), so
// the result is bitwise the one of the stage-wise calls.
template <typename W, bool DIRECT>
__global__ void __launch_bounds__(DIRECT ? 256 : 1024) layer_epilogue_kernel(const EpilogueArgs a) {
    grid_dep_wait();  // the FFN's partial rows
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int q = blockIdx.y * 32 + lane;  // float4 column group
    const int k = a.k, r = a.r, d = a.d, N = a.N;
    const int lore_warp = nw - 1, shared_warp = DIRECT ? nw - 2 : kMaxTopK;
    __shared__ int s_pos[kMaxTopK], s_e[kMaxTopK], s_lore[kMaxTopK], s_kind[kMaxTopK];
    __shared__ float s_g[kMaxTopK];
    __shared__ float s_lg;
    __shared__ int s_nl, s_nslot_u;
    __shared__ int s_slot_unit[kMaxTopK];  // unit of slot s, -1: none (y = 0)
    __shared__ UnitTable U;
    __shared__ float s_z[kMaxTopK * 64];
    __shared__ float4 s_y[kMaxTopK][32];
    __shared__ float4 s_sh[32];
    __shared__ float4 s_yl[32];
    extern __shared__ float4 s_runs[];
    const PlanHeader& hdr = *a.hdr;
    // the segment row of slot s (pos, e), or of shared expert j
    auto slot_seg = [&](int pos, int e, Seg& S, int& row) {
        if (pos < 0 || e < 0 || e >= N || pos >= hdr.n_routed_rows) return false;
        const int local = pos - a.expert_offsets[e];
        const int si = a.seg_first[e] + local / hdr.rg;
        if (si < 0 || si >= hdr.n_seg) return false;
        S = a.segs[si];
        row = local % hdr.rg;
        return seg_row_ok(S, row, hdr.n_partial_rows);
    };
    auto shared_seg = [&](int j, Seg& S, int& row) {
        const int si = a.seg_first[N + j] + t / hdr.rg;
        if (si < 0 || si >= hdr.n_seg) return false;
        S = a.segs[si];
        row = t % hdr.rg;
        return seg_row_ok(S, row, hdr.n_partial_rows);
    };
    if (warp == 0) {
        // lanes 0..k-1: slot s = lane; lanes kMaxTopK..: shared expert lane - kMaxTopK
        const int s = lane;
        bool lore_term = false, has = false;
        Seg S;
        int urow = 0;
        if (s < k) {
            const size_t sl = (size_t)t * k + s;
            const int pos = a.inv_perm[sl];
            const int e = a.final_idx[sl];
            s_pos[s] = pos;
            s_g[s] = a.final_gate[sl];
            s_e[s] = e;
            s_kind[s] = a.final_kind[sl];
            lore_term = s_kind[s] == MOE_KIND_LORE && a.lore_b && e >= 0 && e < N;
            if (!DIRECT) has = slot_seg(pos, e, S, urow);
        } else if (!DIRECT && s >= kMaxTopK && s - kMaxTopK < a.n_shared) {
            has = shared_seg(s - kMaxTopK, S, urow);
        }
        const uint32_t b = __ballot_sync(0xffffffffu, lore_term);
        if (lore_term) s_lore[__popc(b & ((1u << s) - 1u))] = s;
        if (!DIRECT) {
            const int u = unit_table_publish(U, has, S, urow);
            if (s < k) s_slot_unit[s] = u;
        }
        const uint32_t sb = __ballot_sync(0xffffffffu, has && s < kMaxTopK);
        __syncwarp();
        if (s == 0) {  // the LoRE gates summed in slot order
            float lg = 0.f;
            for (int j = 0; j < k; ++j)
                if (s_kind[j] == MOE_KIND_LORE) lg += s_g[j];
            s_lg = lg;
            s_nl = __popc(b);
            s_nslot_u = __popc(sb);
        }
    }
    __syncthreads();
    const bool col_ok = q < d / 4;
    // LoRE term y_lore[t, j] = sum over LoRE slots, then over q, of B_e[j, q] z[q]
    // (the order of lore_b_kernel)
    if (warp == lore_warp && a.lore_b) {
        const int nl = s_nl;
        for (int i = lane; i < nl * r; i += 32) s_z[i] = a.z[((size_t)t * k + s_lore[i / r]) * r + (i % r)];
        __syncwarp();
        float yl[4] = {0.f, 0.f, 0.f, 0.f};
        if (col_ok) {
            const W* B = static_cast<const W*>(a.lore_b);
            constexpr int V = Vec<W>::n;
            const bool vec = (r * (int)sizeof(W)) % 16 == 0;
            for (int i = 0; i < nl; ++i) {
                const int e = s_e[s_lore[i]];
                const float* zz = s_z + i * r;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const W* brow = B + ((size_t)e * d + q * 4 + c) * r;
                    float accl = yl[c];
                    if (vec) {
                        for (int qq = 0; qq < r; qq += V) {
                            float bv[V];
                            unpack16(*reinterpret_cast<const uint4*>(brow + qq), bv, (W*)nullptr);
#pragma unroll
                            for (int u = 0; u < V; ++u) accl = fmaf(bv[u], zz[qq + u], accl);
                        }
                    } else {
                        for (int qq = 0; qq < r; ++qq) accl = fmaf(to_f32(brow[qq]), zz[qq], accl);
                    }
                    yl[c] = accl;
                }
            }
            const float4 v = make_float4(yl[0], yl[1], yl[2], yl[3]);
            reinterpret_cast<float4*>(a.y_lore + (size_t)t * d)[q] = v;
            s_yl[lane] = v;
        }
    }
    if (DIRECT) {
        if (col_ok && warp < k) {
            const int s = warp, pos = s_pos[s];
            if (pos >= 0) {
                Seg S;
                int row = 0;
                const float4 y = slot_seg(pos, s_e[s], S, row) ? partial_unit_sum(a.partial, S, row, d, q)
                                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                reinterpret_cast<float4*>(a.y_perm + (size_t)pos * d)[q] = y;
                s_y[s][lane] = y;
            }
        }
        if (col_ok && warp == shared_warp && a.n_shared > 0) {
            float4 sh = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < a.n_shared; ++j) {
                Seg S;
                int row = 0;
                if (shared_seg(j, S, row)) add4(sh, partial_unit_sum(a.partial, S, row, d, q));
            }
            reinterpret_cast<float4*>(a.y_shared + (size_t)t * d)[q] = sh;
            s_sh[lane] = sh;
        }
    } else {
        if (col_ok && warp != lore_warp) unit_table_runs(U, a.partial, d, q, s_runs, warp, nw - 1);
        __syncthreads();  // the run sums complete
        if (col_ok && warp < k) {
            const int s = warp, pos = s_pos[s];
            if (pos >= 0) {
                const int u = s_slot_unit[s];
                const float4 y = u >= 0 ? unit_table_sum(U, u, s_runs) : make_float4(0.f, 0.f, 0.f, 0.f);
                reinterpret_cast<float4*>(a.y_perm + (size_t)pos * d)[q] = y;
                s_y[s][lane] = y;
            }
        }
        if (col_ok && warp == shared_warp && a.n_shared > 0) {
            float4 sh = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int u = s_nslot_u; u < U.n; ++u) add4(sh, unit_table_sum(U, u, s_runs));
            reinterpret_cast<float4*>(a.y_shared + (size_t)t * d)[q] = sh;
            s_sh[lane] = sh;
        }
    }
    __syncthreads();
    if (warp != 0 || !col_ok) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.n_shared > 0) {
        const float4 sh = s_sh[lane];
        const float scale = 1.f + s_lg;
        acc.x = sh.x * scale; acc.y = sh.y * scale; acc.z = sh.z * scale; acc.w = sh.w * scale;
    }
    for (int s = 0; s < k; ++s) {
        if (s_pos[s] < 0) continue;
        const float4 y = s_y[s][lane];
        const float g = s_g[s];
        acc.x = fmaf(g, y.x, acc.x); acc.y = fmaf(g, y.y, acc.y);
        acc.z = fmaf(g, y.z, acc.z); acc.w = fmaf(g, y.w, acc.w);
    }
    if (a.lore_b) {
        const float4 yl = s_yl[lane];
        acc.x += yl.x; acc.y += yl.y; acc.z += yl.z; acc.w += yl.w;
    }
    reinterpret_cast<float4*>(a.out + (size_t)t * d)[q] = acc;
}

// GEMV partials (segments spread over up to two CTAs per SM, so a token's
// units have up to eight runs each): 32 warps per block share the runs.
// Direct (few pieces per segment): 8 warps.
template <typename K>
static cudaError_t launch_epilogue_k(K kernel, const EpilogueArgs& a, cudaStream_t st) {
    cudaError_t e = allow_max_smem(kernel);
    if (e != cudaSuccess) return e;
    const size_t smem = a.direct ? 0 : (size_t)(a.k + a.n_shared) * kSumChunks * 32 * sizeof(float4);
    const int threads = a.direct ? 256 : 1024;
    dim3 grid(a.T, (a.d / 4 + 31) / 32);
    return launch_pdl(kernel, grid, dim3(threads), smem, st, a);
}

cudaError_t launch_layer_epilogue(const EpilogueArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    if (a.k > kMaxTopK || a.n_shared > kMaxShared) return cudaErrorInvalidValue;
    if (a.direct)
        return a.bf16 ? launch_epilogue_k(layer_epilogue_kernel<__nv_bfloat16, true>, a, st)
                      : launch_epilogue_k(layer_epilogue_kernel<float, true>, a, st);
    return a.bf16 ? launch_epilogue_k(layer_epilogue_kernel<__nv_bfloat16, false>, a, st)
                  : launch_epilogue_k(layer_epilogue_kernel<float, false>, a, st);
}

// One warp waits on a fresh mbarrier (arrival count 1) that no thread ever
// arrives on: the wait gives up after its wall-clock bound and the kernel
// records MOE_ERR_TIMEOUT, as every wait of the library does.
__global__ void wait_timeout_probe_kernel(DevError* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const bool done = mbar_wait(&bar, 0);
    if (!done && threadIdx.x == 0) set_error(err, MOE_ERR_TIMEOUT, -3);
}

cudaError_t launch_wait_timeout_probe(DevError* err, cudaStream_t st) {
    wait_timeout_probe_kernel<<<1, 32, 0, st>>>(err);
    return cudaGetLastError();
}

cudaError_t launch_lore_z(const LoreArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    const dim3 gz(a.T * a.k);
    if (a.bf16)
        lore_z_kernel<__nv_bfloat16><<<gz, 256, 0, st>>>(
            (const __nv_bfloat16*)a.x, a.final_idx, a.final_kind, a.final_gate,
            (const __nv_bfloat16*)a.A, a.d, a.k, a.r, a.N, a.z, a.err);
    else
        lore_z_kernel<float><<<gz, 256, 0, st>>>((const float*)a.x, a.final_idx, a.final_kind,
                                                      a.final_gate, (const float*)a.A, a.d, a.k,
                                                      a.r, a.N, a.z, a.err);
    return cudaGetLastError();
}

cudaError_t launch_lore(const LoreArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    const int n_slots = a.T * a.k;
    const dim3 gz(n_slots);
    dim3 gb(a.T, (a.d + 255) / 256);
    if (a.bf16) {
        lore_z_kernel<__nv_bfloat16><<<gz, 256, 0, st>>>(
            (const __nv_bfloat16*)a.x, a.final_idx, a.final_kind, a.final_gate,
            (const __nv_bfloat16*)a.A, a.d, a.k, a.r, a.N, a.z, a.err);
        lore_b_kernel<__nv_bfloat16><<<gb, 256, 0, st>>>(a.final_idx, a.final_kind,
                                                         (const __nv_bfloat16*)a.B, a.d, a.k, a.r,
                                                         a.N, a.z, a.y_lore);
    } else {
        lore_z_kernel<float><<<gz, 256, 0, st>>>((const float*)a.x, a.final_idx, a.final_kind,
                                                      a.final_gate, (const float*)a.A, a.d, a.k,
                                                      a.r, a.N, a.z, a.err);
        lore_b_kernel<float><<<gb, 256, 0, st>>>(a.final_idx, a.final_kind, (const float*)a.B, a.d,
                                                 a.k, a.r, a.N, a.z, a.y_lore);
    }
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    dim3 grid(a.T, (a.d / 4 + 255) / 256);
    combine_kernel<<<grid, 256, 0, st>>>(a.y_perm, a.inv_perm, a.final_gate, a.final_kind, a.y_shared,
                                        a.y_lore, a.d, a.k, a.out);
    return cudaGetLastError();
}

}  // namespace moe
