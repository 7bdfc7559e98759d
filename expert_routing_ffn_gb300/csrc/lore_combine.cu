// Stages 4 and 5: the SPICE LoRE surrogate residual and the combine.
//
// SPICE write-up, LoRE section: a missing expert e is approximated by
// y_shared + B_e A_e h with A_e [r, d], B_e [d, r], r << d; the shared part
// is added once per token by the combine, scaled by the LoRE slots' gates.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// One block per token: z_s = g_s * A_e x (r dot products of length d, warps
// over rank rows, lanes over d), then y_lore[t, j] = sum_s sum_q B_e[j, q] z_s[q]
// (threads over output columns).  Writes every row (zero without LoRE slots).
template <typename W>
__global__ void __launch_bounds__(256) lore_kernel(const W* __restrict__ x,
                                                   const int32_t* __restrict__ final_idx,
                                                   const int32_t* __restrict__ final_kind,
                                                   const float* __restrict__ final_gate,
                                                   const W* __restrict__ A, const W* __restrict__ B,
                                                   int d, int k, int r, int N,
                                                   float* __restrict__ y_lore,
                                                   DevError* __restrict__ err) {
    constexpr int V = Vec<W>::n;
    extern __shared__ __align__(16) float lsm[];
    float* xs = lsm;               // [d]
    float* zs = lsm + d;           // [k][r]
    __shared__ int s_e[kMaxTopK];
    __shared__ float s_gate[kMaxTopK];
    __shared__ int s_n;
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    if (tid == 0) {
        int n = 0;
        for (int s = 0; s < k; ++s) {
            const size_t sl = (size_t)t * k + s;
            if (final_kind[sl] == MOE_KIND_LORE) {
                const int e = final_idx[sl];
                if (e < 0 || e >= N) { if (err) set_error(err, MOE_ERR_DEVICE_INDEX, (int)sl); continue; }
                s_e[n] = e;
                s_gate[n] = final_gate[sl];
                ++n;
            }
        }
        s_n = n;
    }
    __syncthreads();
    const int n = s_n;
    if (n == 0) {
        for (int j = tid; j < d; j += blockDim.x) y_lore[(size_t)t * d + j] = 0.f;
        return;
    }
    for (int j = tid; j < d; j += blockDim.x) xs[j] = to_f32(x[(size_t)t * d + j]);
    __syncthreads();
    const int nchunk = d / V;
    for (int job = warp; job < n * r; job += nw) {
        const int s = job / r, q = job % r;
        const W* arow = A + ((size_t)s_e[s] * r + q) * d;
        float acc = 0.f;
        for (int c = lane; c < nchunk; c += 32) {
            float av[V];
            unpack16(reinterpret_cast<const uint4*>(arow)[c], av, (W*)nullptr);
#pragma unroll
            for (int j = 0; j < V; ++j) acc = fmaf(av[j], xs[c * V + j], acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) zs[s * r + q] = s_gate[s] * acc;
    }
    __syncthreads();
    for (int j = tid; j < d; j += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < n; ++s) {
            const W* brow = B + ((size_t)s_e[s] * d + j) * r;
            for (int q = 0; q < r; ++q) acc = fmaf(to_f32(brow[q]), zs[s * r + q], acc);
        }
        y_lore[(size_t)t * d + j] = acc;
    }
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
    const int nd4 = d / 4;
    for (int q = threadIdx.x; q < nd4; q += blockDim.x) {
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
    const size_t smem = ((size_t)a.d + (size_t)kMaxTopK * a.r) * sizeof(float);
    if (a.bf16) {
        if (smem > 48 * 1024 && allow_max_smem(lore_kernel<__nv_bfloat16>) != cudaSuccess)
            return cudaErrorInvalidValue;
        lore_kernel<__nv_bfloat16><<<a.T, 256, smem, st>>>(
            (const __nv_bfloat16*)a.x, a.final_idx, a.final_kind, a.final_gate,
            (const __nv_bfloat16*)a.A, (const __nv_bfloat16*)a.B, a.d, a.k, a.r, a.N, a.y_lore, a.err);
    } else {
        if (smem > 48 * 1024 && allow_max_smem(lore_kernel<float>) != cudaSuccess)
            return cudaErrorInvalidValue;
        lore_kernel<float><<<a.T, 256, smem, st>>>((const float*)a.x, a.final_idx, a.final_kind,
                                                   a.final_gate, (const float*)a.A, (const float*)a.B,
                                                   a.d, a.k, a.r, a.N, a.y_lore, a.err);
    }
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    combine_kernel<<<a.T, 256, 0, st>>>(a.y_perm, a.inv_perm, a.final_gate, a.final_kind, a.y_shared,
                                        a.y_lore, a.d, a.k, a.out);
    return cudaGetLastError();
}

}  // namespace moe
