// Confidence-aware prefetch depth over J look-ahead layers.
//
// SPICE write-up, section on confidence-aware adaptive prefetch: a draft
// predicts the expert distribution of each of the next layers from the
// current hidden state; its confidence is the probability mass on the
// predicted top-K experts; prediction goes one layer deeper while the
// confidence stays at or above the threshold and stops at the first layer
// below it; the depth is never less than the minimum depth D_min that hides a
// transfer behind the layers it runs ahead of.  The look-ahead routers'
// logits come from one launch below for decode-size batches, else from the
// router GEMM paths (route.cu, route_tc.cu); the depth kernel reads them,
// [J][T][N] fp32:
//   conf[t][j]  = sum of softmax over the K largest logits (ties: lower index)
//   depth[t]    = min(J, max(d_min, c)), c = leading layers with conf >= tau
//   tok[t][j]   = the top-K set of layer j for j < depth[t], else 0
//   layer[j]   |= tok[t][j]      (layer masks zeroed before the launch)
// A warp per (token, layer), N <= 64 (two logits per lane); the block ORs
// its tokens' sets in shared memory and adds them to the layer masks with one
// atomic per layer.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kAheadTT = 8;  // tokens per block of the look-ahead logits

// ---------------------------------------------------------------- logits
// Decode-size batches: the logits of all J look-ahead routers in one launch,
// which also zeroes the layer masks for the depth launch.
// Block (token tile, 8 router rows of the J*N stacked rows): the tile's x rows
// staged in shared memory, a warp per router row streaming it once in
// 16-byte chunks (lane-strided) against every token of the tile.
struct AheadRouters {
    const void* w[kMaxAhead];   // [N, d] per look-ahead layer
    const float* b[kMaxAhead];  // [N] or NULL
};

__device__ __forceinline__ void ahead_unpack(const uint4& v, float* f, const __nv_bfloat16*) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 p = __bfloat1622float2(h[i]);
        f[2 * i] = p.x;
        f[2 * i + 1] = p.y;
    }
}
__device__ __forceinline__ void ahead_unpack(const uint4& v, float* f, const float*) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y); f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}

template <typename W>
__global__ void __launch_bounds__(256) lookahead_logits_kernel(const W* __restrict__ x, const AheadRouters R, int T,
                                                              int d, int N, int J, float* __restrict__ logits,
                                                              unsigned long long* __restrict__ layer_masks) {
    grid_dep_wait();  // x comes from the previous launches
    // the depth launch that follows ORs into the layer masks
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < J) layer_masks[threadIdx.x] = 0ull;
    const int rows = J * N;
    extern __shared__ __align__(16) unsigned char ahead_smem[];
    constexpr int EPC = 16 / (int)sizeof(W);  // values per 16-byte chunk
    const int cpr = d / EPC;
    const int t0 = blockIdx.x * kAheadTT;
    const int nt = T - t0 < kAheadTT ? T - t0 : kAheadTT;
    uint4* xs = reinterpret_cast<uint4*>(ahead_smem);
    const uint4* xg = reinterpret_cast<const uint4*>(x + (size_t)t0 * d);
    for (int i = threadIdx.x; i < nt * cpr; i += blockDim.x) xs[i] = xg[i];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.y * 8 + warp;
    if (r >= rows) return;
    const int j = r / N, e = r % N;
    const uint4* w = reinterpret_cast<const uint4*>(static_cast<const W*>(R.w[j]) + (size_t)e * d);
    float acc[kAheadTT];
#pragma unroll
    for (int tt = 0; tt < kAheadTT; ++tt) acc[tt] = 0.f;
#pragma unroll 4
    for (int c = lane; c < cpr; c += 32) {
        float wf[EPC];
        ahead_unpack(w[c], wf, static_cast<const W*>(nullptr));
#pragma unroll
        for (int tt = 0; tt < kAheadTT; ++tt) {
            if (tt < nt) {
                float xf[EPC];
                ahead_unpack(xs[tt * cpr + c], xf, static_cast<const W*>(nullptr));
#pragma unroll
                for (int q = 0; q < EPC; ++q) acc[tt] = fmaf(wf[q], xf[q], acc[tt]);
            }
        }
    }
#pragma unroll
    for (int tt = 0; tt < kAheadTT; ++tt)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[tt] += __shfl_xor_sync(0xffffffffu, acc[tt], o);
    if (lane == 0) {
        const float bias = R.b[j] ? R.b[j][e] : 0.f;
        for (int tt = 0; tt < nt; ++tt) logits[((size_t)j * T + t0 + tt) * N + e] = acc[tt] + bias;
    }
}

cudaError_t launch_lookahead_logits(const void* x, const void* const* w, const float* const* b, int J, int T, int d,
                                    int N, bool bf16, float* logits, uint64_t* layer_masks, cudaStream_t st) {
    AheadRouters R;
    for (int j = 0; j < kMaxAhead; ++j) {
        R.w[j] = j < J ? w[j] : nullptr;
        R.b[j] = (j < J && b) ? b[j] : nullptr;
    }
    const int rows = J * N;
    const dim3 grid((T + kAheadTT - 1) / kAheadTT, (rows + 7) / 8);
    const size_t smem = (size_t)kAheadTT * d * (bf16 ? 2 : 4);
    if (bf16) {
        cudaError_t e = allow_max_smem(lookahead_logits_kernel<__nv_bfloat16>);
        if (e != cudaSuccess) return e;
        return launch_pdl(lookahead_logits_kernel<__nv_bfloat16>, grid, dim3(256), smem, st,
                          static_cast<const __nv_bfloat16*>(x), R, T, d, N, J, logits,
                          reinterpret_cast<unsigned long long*>(layer_masks));
    }
    cudaError_t e = allow_max_smem(lookahead_logits_kernel<float>);
    if (e != cudaSuccess) return e;
    return launch_pdl(lookahead_logits_kernel<float>, grid, dim3(256), smem, st, static_cast<const float*>(x), R, T, d,
                      N, J, logits, reinterpret_cast<unsigned long long*>(layer_masks));
}

// ---------------------------------------------------------------- depth
// (v, i) ranks above (w, k): larger logit, or equal and lower index
__device__ __forceinline__ bool ahead_above(float v, int i, float w, int k) { return v > w || (v == w && i < k); }

// Block: tpb = max(1, 16 / J) tokens, a warp per (token, look-ahead layer)
// pair for the softmax and the top-K (K rounds of a warp arg-max), then a
// thread per token for the depth scan and the masks; the block's sets are
// OR-ed in shared memory and reach the layer masks with one atomic per layer.
__global__ void __launch_bounds__(32 * kMaxAhead) prefetch_depth_kernel(
    const float* __restrict__ logits, int T, int N, int K, int J, int tpb, float tau, int d_min,
    float* __restrict__ conf, int32_t* __restrict__ depth, uint64_t* __restrict__ tok_masks,
    unsigned long long* __restrict__ layer_masks) {
    grid_dep_wait();  // the look-ahead logits come from the previous launches
    __shared__ float s_conf[kMaxAhead];
    __shared__ unsigned long long s_set[kMaxAhead], s_or[kMaxAhead];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x < kMaxAhead) s_or[threadIdx.x] = 0ull;
    const int lt = warp / J, j = warp % J;  // this warp's token (in the block) and layer
    const int t = blockIdx.x * tpb + lt;
    if (lt < tpb && t < T) {
        const float* l = logits + ((size_t)j * T + t) * N;
        const int i0 = lane, i1 = lane + 32;
        const float v0 = i0 < N ? l[i0] : -INFINITY;
        const float v1 = i1 < N ? l[i1] : -INFINITY;
        float m = fmaxf(v0, v1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float s = (i0 < N ? expf(v0 - m) : 0.f) + (i1 < N ? expf(v1 - m) : 0.f);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        // K rounds of a warp arg-max over the experts not yet taken
        bool t0 = i0 >= N, t1 = i1 >= N;
        float mass = 0.f;
        unsigned long long set = 0ull;
        for (int r = 0; r < K; ++r) {
            float bv = -INFINITY;
            int bi = 1 << 30;
            if (!t0) { bv = v0; bi = i0; }
            if (!t1 && ahead_above(v1, i1, bv, bi)) { bv = v1; bi = i1; }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ahead_above(ov, oi, bv, bi)) { bv = ov; bi = oi; }
            }
            if (bi == i0) t0 = true;
            if (bi == i1) t1 = true;
            mass += expf(bv - m);
            set |= 1ull << bi;
        }
        if (lane == 0) {
            const float cf = mass / s;
            conf[(size_t)t * J + j] = cf;
            s_conf[warp] = cf;
            s_set[warp] = set;
        }
    }
    __syncthreads();
    const int tt = threadIdx.x, tok = blockIdx.x * tpb + tt;
    if (tt < tpb && tok < T) {
        int c = 0;
        while (c < J && s_conf[tt * J + c] >= tau) ++c;
        int dep = c > d_min ? c : d_min;
        if (dep > J) dep = J;
        depth[tok] = dep;
        for (int q = 0; q < J; ++q) {
            const unsigned long long sq = q < dep ? s_set[tt * J + q] : 0ull;
            tok_masks[(size_t)tok * J + q] = sq;
            if (sq) atomicOr(&s_or[q], sq);
        }
    }
    __syncthreads();
    if (threadIdx.x < J && s_or[threadIdx.x]) atomicOr(&layer_masks[threadIdx.x], s_or[threadIdx.x]);
}

cudaError_t launch_prefetch_depth(const float* logits, int T, int N, int K, int J, float tau, int d_min,
                                  float* conf, int32_t* depth, uint64_t* tok_masks, uint64_t* layer_masks,
                                  cudaStream_t st) {
    const int tpb = J >= kMaxAhead ? 1 : kMaxAhead / J;  // tokens per block: tpb * J <= 16 warps
    const int blocks = (T + tpb - 1) / tpb;
    return launch_pdl(prefetch_depth_kernel, dim3(blocks), dim3(32 * tpb * J), 0, st, logits, T, N, K, J, tpb, tau,
                      d_min, conf, depth, tok_masks, reinterpret_cast<unsigned long long*>(layer_masks));
}

}  // namespace moe
