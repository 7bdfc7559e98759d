// Stages 4 and 5: the SPICE LoRE surrogate residual and the combine.
//
// SPICE write-up, LoRE section: a missing expert e is approximated by
// y_shared + B_e A_e h with A_e [r, d], B_e [d, r], r << d; the shared part
// is added once per token by the combine, scaled by the LoRE slots' gates.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// z[t, s, :] = g_s * A_e x_t for a LoRE slot (t, s) (zero for other slots):
// one block per slot, warps over the r rank rows, lanes over d.
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
    const int q_begin = blockIdx.y * nw, q_end = min(r, q_begin + nw);  // one rank row per warp
    const int e = final_idx[slot];
    if (final_kind[slot] != MOE_KIND_LORE || e < 0 || e >= N) {
        if (final_kind[slot] == MOE_KIND_LORE && err && tid == 0 && blockIdx.y == 0)
            set_error(err, MOE_ERR_DEVICE_INDEX, slot);
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
    if (threadIdx.x == 0) {
        int n = 0;
        for (int s = 0; s < k; ++s) {
            const size_t sl = (size_t)t * k + s;
            const int e = final_idx[sl];
            if (final_kind[sl] == MOE_KIND_LORE && e >= 0 && e < N) s_e[n++] = s;
        }
        s_n = n;
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
    __shared__ int s_pos[kMaxTopK];
    __shared__ float s_g[kMaxTopK];
    __shared__ float s_lg;
    if (threadIdx.x == 0) {
        float lg = 0.f;
        for (int s = 0; s < k; ++s) {
            const size_t sl = (size_t)t * k + s;
            s_pos[s] = inv_perm[sl];
            s_g[s] = final_gate[sl];
            if (final_kind[sl] == MOE_KIND_LORE) lg += final_gate[sl];
        }
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

cudaError_t launch_lore(const LoreArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    const int n_slots = a.T * a.k;
    dim3 gz(n_slots, (a.r + 3) / 4);  // 4 warps = 4 rank rows per block
    dim3 gb(a.T, (a.d + 255) / 256);
    if (a.bf16) {
        lore_z_kernel<__nv_bfloat16><<<gz, 128, 0, st>>>(
            (const __nv_bfloat16*)a.x, a.final_idx, a.final_kind, a.final_gate,
            (const __nv_bfloat16*)a.A, a.d, a.k, a.r, a.N, a.z, a.err);
        lore_b_kernel<__nv_bfloat16><<<gb, 256, 0, st>>>(a.final_idx, a.final_kind,
                                                         (const __nv_bfloat16*)a.B, a.d, a.k, a.r,
                                                         a.N, a.z, a.y_lore);
    } else {
        lore_z_kernel<float><<<gz, 128, 0, st>>>((const float*)a.x, a.final_idx, a.final_kind,
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
