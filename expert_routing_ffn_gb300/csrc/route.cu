// Stage 1 and 2 kernels: router / prefetch-router logits, per-token warp
// selection (softmax, top-k, ordinal-CDF budget, prefetch set, delta*), the
// batch resident set, and the per-token miss handling (stall-free
// substitution, LoRE, fetch).
//
// APEX: Adaptive Expert Prefetching for Edge MoE Inference — §4.1 (prefetch
// router: linear + softmax on the pre-attention state), §4.2 (delta*,
// p_delta = sigmoid(theta_delta - w.x), delta_hat = min{delta : p_delta >=
// tau}), §4.3 (Algorithm 1 stall_free_select; correctness-preserving mode).
// SPICE write-up, LoRE section: low-confidence misses use the surrogate.
#include "common.cuh"
#include "kernels.h"
#include "plan.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Logits: one warp per output row o (router rows 0..N-1 on x, prefetch rows
// N..2N-1 and the ordinal scorer row 2N on x_pre), for a tile of TT tokens.
// Lanes split d in 16-byte chunks; each lane sums its chunk products in order
// and the warp adds the 32 partial sums as a tree, which keeps the fp32
// rounding error of a logit near 1e-7 (the decisions made on these logits are
// compared bit-exactly with a float64 reference, away from near-ties).
template <typename W, int TT>
__device__ __forceinline__ void logits_tile(
    const W* __restrict__ x, const W* __restrict__ x_pre, const W* __restrict__ w_router,
    const float* __restrict__ bias, const W* __restrict__ w_prefetch, const float* __restrict__ w_ord,
    int T, int d, int N, int n_out, int rows_per_block, float* __restrict__ logits_r,
    float* __restrict__ logits_p, float* __restrict__ score, unsigned char* smem_raw) {
    constexpr int V = Vec<W>::n;
    W* xs = reinterpret_cast<W*>(smem_raw);                 // [TT][d]
    W* xps = xs + (size_t)TT * d;                             // [TT][d] (x_pre)
    const int t0 = blockIdx.x * TT;
    const int nt = min(TT, T - t0);
    const int nchunk = d / V;
    const bool sep = (x_pre != x);
    // stage the token tile (16-byte copies, eight loads in flight per thread)
    constexpr int U = 8;
    for (int i0 = threadIdx.x; i0 < TT * nchunk; i0 += blockDim.x * U) {
        uint4 v[U], vp[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * blockDim.x;
            const int t = i / nchunk, q = i % nchunk;
            v[u] = make_uint4(0, 0, 0, 0);
            vp[u] = make_uint4(0, 0, 0, 0);
            if (i < TT * nchunk && t < nt) {
                v[u] = reinterpret_cast<const uint4*>(x + (size_t)(t0 + t) * d)[q];
                if (sep) vp[u] = reinterpret_cast<const uint4*>(x_pre + (size_t)(t0 + t) * d)[q];
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * blockDim.x;
            if (i < TT * nchunk) {
                const int t = i / nchunk, q = i % nchunk;
                reinterpret_cast<uint4*>(xs + (size_t)t * d)[q] = v[u];
                if (sep) reinterpret_cast<uint4*>(xps + (size_t)t * d)[q] = vp[u];
            }
        }
    }
    __syncthreads();
    const W* xsp = sep ? xps : xs;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int o_begin = blockIdx.y * rows_per_block;
    const int o_end = min(n_out, o_begin + rows_per_block);
    for (int o = o_begin + warp; o < o_end; o += nw) {
        const W* wrow;
        const W* tile;
        bool is_ord = false;
        if (o < N) { wrow = w_router + (size_t)o * d; tile = xs; }
        else if (o < 2 * N) { wrow = w_prefetch + (size_t)(o - N) * d; tile = xsp; }
        else { wrow = nullptr; tile = xsp; is_ord = true; }
        float acc[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[t] = 0.f;
        // the lane's weight chunks q = lane, lane + 32, ... in groups of QU,
        // all loads of a group in flight before the products (same order of
        // accumulation as one chunk at a time)
        constexpr int QU = 8;
        for (int q0 = lane; q0 < nchunk; q0 += 32 * QU) {
            uint4 wraw[QU];
            if (!is_ord) {
#pragma unroll
                for (int u = 0; u < QU; ++u) {
                    const int q = q0 + 32 * u;
                    wraw[u] = q < nchunk ? reinterpret_cast<const uint4*>(wrow)[q] : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int u = 0; u < QU; ++u) {
                const int q = q0 + 32 * u;
                if (q >= nchunk) break;
                float wv[V];
                if (!is_ord) {
                    unpack16(wraw[u], wv, (W*)nullptr);
                } else {
#pragma unroll
                    for (int j = 0; j < V; ++j) wv[j] = w_ord[q * V + j];
                }
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    uint4 raw = reinterpret_cast<const uint4*>(tile + (size_t)t * d)[q];
                    float xv[V];
                    unpack16(raw, xv, (W*)nullptr);
#pragma unroll
                    for (int j = 0; j < V; ++j) acc[t] = fmaf(xv[j], wv[j], acc[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[t] = warp_sum(acc[t]);
        if (lane == 0) {
            for (int t = 0; t < nt; ++t) {
                const int tok = t0 + t;
                if (o < N) logits_r[(size_t)tok * N + o] = acc[t] + (bias ? bias[o] : 0.f);
                else if (o < 2 * N) logits_p[(size_t)tok * N + (o - N)] = acc[t];
                else score[tok] = acc[t];
            }
        }
    }
}

template <typename W, int TT>
__global__ void __launch_bounds__(256) route_logits_kernel(
    const W* __restrict__ x, const W* __restrict__ x_pre, const W* __restrict__ w_router,
    const float* __restrict__ bias, const W* __restrict__ w_prefetch, const float* __restrict__ w_ord,
    int T, int d, int N, int n_out, int rows_per_block, float* __restrict__ logits_r,
    float* __restrict__ logits_p, float* __restrict__ score) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    logits_tile<W, TT>(x, x_pre, w_router, bias, w_prefetch, w_ord, T, d, N, n_out, rows_per_block, logits_r,
                       logits_p, score, smem_raw);
}

// Large batches: a register-tiled version of the same logits.  Block tile =
// 64 tokens x 64 output rows, K in chunks of 32 through shared memory (fp32,
// x stored K-major so a thread reads 4 tokens with one 16-byte load).  Each
// thread owns 4 tokens x 4 rows.  Every chunk's 32 products are summed into a
// fresh partial that is then added to the running total (blocked summation),
// keeping the rounding error of a logit near 1e-7.
template <typename W>
__global__ void __launch_bounds__(256) route_logits_tiled_kernel(
    const W* __restrict__ x, const W* __restrict__ x_pre, const W* __restrict__ w_router,
    const float* __restrict__ bias, const W* __restrict__ w_prefetch, const float* __restrict__ w_ord,
    int T, int d, int N, int n_out, float* __restrict__ logits_r, float* __restrict__ logits_p,
    float* __restrict__ score) {
    constexpr int TT = 64, TO = 64, KC = 32;
    constexpr int V = Vec<W>::n;
    constexpr int XL = TT * KC / V / 256;  // 16-byte loads per thread per chunk (token tiles)
    constexpr int WL = TO * KC / V / 256;  // (weight rows)
    static_assert(XL >= 1 && WL >= 1, "tile and chunk sizes");
    __shared__ __align__(16) float xs[KC][TT];    // router input x
    __shared__ __align__(16) float xps[KC][TT];   // prefetch input x_pre
    __shared__ __align__(16) float ws[KC][TO];
    const int t0 = blockIdx.x * TT, o0 = blockIdx.y * TO;
    const int tid = threadIdx.x;
    const int tq = tid & 15, oq = tid >> 4;       // 16 token quads x 16 row quads
    const bool sep = x_pre != x;
    const int n_rows = 2 * N;                     // router rows, then prefetch rows (the scorer runs apart)
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
    // the next chunk's global loads, issued before the current chunk's products
    uint4 rx[XL], rxp[XL], rw[WL];
    auto load = [&](int k0) {
#pragma unroll
        for (int j = 0; j < XL; ++j) {
            const int i = tid + j * 256;
            const int tt = i / (KC / V), kv = (i % (KC / V)) * V, tok = t0 + tt;
            rx[j] = make_uint4(0, 0, 0, 0);
            rxp[j] = make_uint4(0, 0, 0, 0);
            if (tok < T) {
                rx[j] = *reinterpret_cast<const uint4*>(x + (size_t)tok * d + k0 + kv);
                if (sep) rxp[j] = *reinterpret_cast<const uint4*>(x_pre + (size_t)tok * d + k0 + kv);
            }
        }
#pragma unroll
        for (int j = 0; j < WL; ++j) {
            const int i = tid + j * 256;
            const int oo = i / (KC / V), kv = (i % (KC / V)) * V, o = o0 + oo;
            rw[j] = make_uint4(0, 0, 0, 0);
            if (o < N) rw[j] = *reinterpret_cast<const uint4*>(w_router + (size_t)o * d + k0 + kv);
            else if (o < n_rows) rw[j] = *reinterpret_cast<const uint4*>(w_prefetch + (size_t)(o - N) * d + k0 + kv);
        }
    };
    load(0);
    for (int k0 = 0; k0 < d; k0 += KC) {
        // registers -> K-major shared tiles (fp32)
#pragma unroll
        for (int j = 0; j < XL; ++j) {
            const int i = tid + j * 256;
            const int tt = i / (KC / V), kv = (i % (KC / V)) * V;
            float v[V], vp[V];
            unpack16(rx[j], v, (W*)nullptr);
            unpack16(rxp[j], vp, (W*)nullptr);
#pragma unroll
            for (int u = 0; u < V; ++u) {
                xs[kv + u][tt] = v[u];
                xps[kv + u][tt] = sep ? vp[u] : v[u];
            }
        }
#pragma unroll
        for (int j = 0; j < WL; ++j) {
            const int i = tid + j * 256;
            const int oo = i / (KC / V), kv = (i % (KC / V)) * V;
            float v[V];
            unpack16(rw[j], v, (W*)nullptr);
#pragma unroll
            for (int u = 0; u < V; ++u) ws[kv + u][oo] = v[u];
        }
        __syncthreads();
        if (k0 + KC < d) load(k0 + KC);
        float part[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) part[a][b] = 0.f;
        // rows o < N use x, the prefetch rows use x_pre
        const bool pre = o0 + oq * 4 >= N;
#pragma unroll 8
        for (int kk = 0; kk < KC; ++kk) {
            const float4 xv = *reinterpret_cast<const float4*>(pre ? &xps[kk][tq * 4] : &xs[kk][tq * 4]);
            const float4 wv = *reinterpret_cast<const float4*>(&ws[kk][oq * 4]);
            const float xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; b += 2)
                    fma2(part[a][b], part[a][b + 1], xa[a], xa[a], wa[b], wa[b + 1]);
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] += part[a][b];
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int tok = t0 + tq * 4 + a;
        if (tok >= T) continue;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int o = o0 + oq * 4 + b;
            if (o < N) logits_r[(size_t)tok * N + o] = acc[a][b] + (bias ? bias[o] : 0.f);
            else if (o < n_rows) logits_p[(size_t)tok * N + (o - N)] = acc[a][b];
        }
    }
    (void)n_out;
    (void)w_ord;
    (void)score;
}

// The ordinal scorer s = w . x_pre for large batches: one warp per token,
// lanes over 16-byte chunks of d, each lane's products in order, then a warp
// tree (the accumulation of route_logits_kernel).
template <typename W>
__global__ void __launch_bounds__(256) route_score_kernel(const W* __restrict__ x_pre,
                                                          const float* __restrict__ w_ord, int T, int d,
                                                          float* __restrict__ score) {
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
    constexpr int V = Vec<W>::n;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const uint4* xr = reinterpret_cast<const uint4*>(x_pre + (size_t)t * d);
    float acc = 0.f;
    int q = lane;
    if ((reinterpret_cast<uintptr_t>(w_ord) & 15) == 0) {
        // four chunks per lane in flight (x and w loaded before the products,
        // which keep the order of the loop below)
        const float4* w4 = reinterpret_cast<const float4*>(w_ord);
        for (; q + 96 < d / V; q += 128) {
            uint4 xa[4];
            float4 wa[4][V / 4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                xa[u] = xr[q + 32 * u];
#pragma unroll
                for (int i = 0; i < V / 4; ++i) wa[u][i] = w4[(q + 32 * u) * (V / 4) + i];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float xv[V];
                unpack16(xa[u], xv, (W*)nullptr);
                const float* wv = reinterpret_cast<const float*>(wa[u]);
#pragma unroll
                for (int j = 0; j < V; ++j) acc = fmaf(xv[j], wv[j], acc);
            }
        }
    }
    for (; q < d / V; q += 32) {
        float xv[V];
        unpack16(xr[q], xv, (W*)nullptr);
#pragma unroll
        for (int j = 0; j < V; ++j) acc = fmaf(xv[j], w_ord[q * V + j], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) score[t] = acc;
}

// (value, index) argmax across the warp: larger value wins, equal values go
// to the lower index.  Lanes with no candidate pass index = INT_MAX.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, v, o);
        int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
    }
}

// best of this lane's two candidates (experts lane, lane + 32) within `mask`
__device__ __forceinline__ void lane_best(float v0, float v1, uint64_t mask, int lane, float& v, int& i) {
    v = -INFINITY;
    i = 0x7fffffff;
    if ((mask >> lane) & 1) { v = v0; i = lane; }
    if ((mask >> (lane + 32)) & 1) {
        if (i == 0x7fffffff || v1 > v) { v = v1; i = lane + 32; }
    }
}

__device__ __forceinline__ uint64_t valid_mask(int N) {
    return N >= 64 ? ~0ull : ((1ull << N) - 1ull);
}

// ---------------------------------------------------------------------------
// One warp per token: softmax, top-k, delta_hat, prefetch set, delta*.
__device__ __forceinline__ void route_select_token(
    int t, const float* __restrict__ logits_r, const float* __restrict__ logits_p,
    const float* __restrict__ score, const float* __restrict__ theta, float logit_tau,
    int N, int k, int delta_max, int has_prefetch, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_gate, float* __restrict__ router_prob, int32_t* __restrict__ delta_hat,
    uint64_t* __restrict__ prefetch_mask, int32_t* __restrict__ delta_star, float* __restrict__ qp) {
    const int lane = threadIdx.x & 31;
    const int e0 = lane, e1 = lane + 32;
    const float l0 = e0 < N ? logits_r[(size_t)t * N + e0] : -INFINITY;
    const float l1 = e1 < N ? logits_r[(size_t)t * N + e1] : -INFINITY;
    const float q0 = has_prefetch && e0 < N ? logits_p[(size_t)t * N + e0] : -INFINITY;
    const float q1 = has_prefetch && e1 < N ? logits_p[(size_t)t * N + e1] : -INFINITY;
    // softmax
    const float m = warp_max(fmaxf(l0, l1));
    const float p0 = e0 < N ? expf(l0 - m) : 0.f;
    const float p1 = e1 < N ? expf(l1 - m) : 0.f;
    const float s = warp_sum(p0 + p1);
    const float a0 = p0 / s, a1 = p1 / s;
    if (e0 < N) router_prob[(size_t)t * N + e0] = a0;
    if (e1 < N) router_prob[(size_t)t * N + e1] = a1;
    // Ranks in descending order, lowest index first on ties, of the router
    // logits (g) and the prefetch logits (r): the number of experts ahead of
    // e0 / e1.  One pass of independent comparisons, eight shuffles in flight
    // (experts past N hold -inf and are never ahead).
    int g0 = 0, g1 = 0, r0 = 0, r1 = 0;
#pragma unroll 8
    for (int j = 0; j < 64; ++j) {
        const float lj = __shfl_sync(0xffffffffu, j < 32 ? l0 : l1, j & 31);
        const float qj = __shfl_sync(0xffffffffu, j < 32 ? q0 : q1, j & 31);
        g0 += (lj > l0 || (lj == l0 && j < e0)) ? 1 : 0;
        g1 += (lj > l1 || (lj == l1 && j < e1)) ? 1 : 0;
        r0 += (qj > q0 || (qj == q0 && j < e0)) ? 1 : 0;
        r1 += (qj > q1 || (qj == q1 && j < e1)) ? 1 : 0;
    }
    // top-k of the logits: the experts of rank < k, each at its rank
    const bool tk0 = e0 < N && g0 < k, tk1 = e1 < N && g1 < k;
    if (tk0) { topk_idx[(size_t)t * k + g0] = e0; topk_gate[(size_t)t * k + g0] = a0; }
    if (tk1) { topk_idx[(size_t)t * k + g1] = e1; topk_gate[(size_t)t * k + g1] = a1; }
    const uint64_t routed = (uint64_t)__ballot_sync(0xffffffffu, tk0) |
                            ((uint64_t)__ballot_sync(0xffffffffu, tk1) << 32);
    if (!has_prefetch) {
        if (lane == 0) {
            delta_hat[t] = 0;
            prefetch_mask[t] = ~0ull;
            if (delta_star) delta_star[t] = 0;
        }
        return;
    }
    // delta_hat = smallest delta with theta_delta - s >= logit(tau)
    // (the same test as sigmoid(theta_delta - s) >= tau; sigmoid is monotone)
    const float sc = score[t];
    const bool c0 = lane <= delta_max && (theta[lane] - sc) >= logit_tau;
    const bool c1 = lane + 32 <= delta_max && (theta[lane + 32] - sc) >= logit_tau;
    const uint32_t b0 = __ballot_sync(0xffffffffu, c0), b1 = __ballot_sync(0xffffffffu, c1);
    int dh = delta_max;
    if (b0) dh = __ffs(b0) - 1;
    else if (b1) dh = 32 + __ffs(b1) - 1;
    dh = min(dh, delta_max);
    const int lim = k + dh;
    const uint32_t in0 = __ballot_sync(0xffffffffu, e0 < N && r0 < lim);
    const uint32_t in1 = __ballot_sync(0xffffffffu, e1 < N && r1 < lim);
    const uint64_t pm = (uint64_t)in0 | ((uint64_t)in1 << 32);
    // delta* = max(0, max over routed experts of rank_p + 1 - k)
    int worst = -1;
    if ((routed >> e0) & 1) worst = max(worst, r0);
    if ((routed >> e1) & 1) worst = max(worst, r1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) worst = max(worst, __shfl_xor_sync(0xffffffffu, worst, o));
    if (lane == 0) {
        delta_hat[t] = dh;
        prefetch_mask[t] = pm;
        if (delta_star) delta_star[t] = max(0, worst + 1 - k);
    }
    if (qp) {
        const float mq = warp_max(fmaxf(q0, q1));
        const float z0 = e0 < N ? expf(q0 - mq) : 0.f;
        const float z1 = e1 < N ? expf(q1 - mq) : 0.f;
        const float zs = warp_sum(z0 + z1);
        if (e0 < N) qp[(size_t)t * N + e0] = z0 / zs;
        if (e1 < N) qp[(size_t)t * N + e1] = z1 / zs;
    }
}

__global__ void __launch_bounds__(256) route_select_kernel(
    const float* __restrict__ logits_r, const float* __restrict__ logits_p,
    const float* __restrict__ score, const float* __restrict__ theta, float logit_tau, int T,
    int N, int k, int delta_max, int has_prefetch, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_gate, float* __restrict__ router_prob, int32_t* __restrict__ delta_hat,
    uint64_t* __restrict__ prefetch_mask, int32_t* __restrict__ delta_star, float* __restrict__ qp) {
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp >= T) return;
    route_select_token(warp, logits_r, logits_p, score, theta, logit_tau, N, k, delta_max, has_prefetch,
                       topk_idx, topk_gate, router_prob, delta_hat, prefetch_mask, delta_star, qp);
}

// ---------------------------------------------------------------------------
// Batch resident set: the n_res experts with the largest prefetch probability
// summed over the tokens, in a fixed summation order (16 token groups per
// expert, then the groups in order; any block size).
__device__ __forceinline__ void batch_resident_block(const float* __restrict__ qp, int T, int N, int n_res,
                                                     uint64_t* __restrict__ out) {
    __shared__ float part[16][64];
    __shared__ float tot[64];
    __shared__ uint32_t bits[2];
    for (int idx = threadIdx.x; idx < 16 * 64; idx += blockDim.x) {
        const int e = idx & 63, g = idx >> 6;
        float acc = 0.f;
        if (e < N)
            for (int t = g; t < T; t += 16) acc += qp[(size_t)t * N + e];
        part[g][e] = acc;
    }
    __syncthreads();
    if (threadIdx.x < 64) {
        float s = 0.f;
        for (int i = 0; i < 16; ++i) s += part[i][threadIdx.x];
        tot[threadIdx.x] = s;
    }
    __syncthreads();
    if (threadIdx.x < 64) {
        const int me = threadIdx.x;
        int rank = 0;
        if (me < N) {
            for (int j = 0; j < N; ++j)
                rank += (tot[j] > tot[me] || (tot[j] == tot[me] && j < me)) ? 1 : 0;
        }
        const uint32_t b = __ballot_sync(0xffffffffu, me < N && rank < n_res);
        if ((me & 31) == 0) bits[me >> 5] = b;
    }
    __syncthreads();
    if (threadIdx.x == 0) *out = (uint64_t)bits[0] | ((uint64_t)bits[1] << 32);
}

__global__ void __launch_bounds__(1024) batch_resident_kernel(const float* __restrict__ qp, int T,
                                                              int N, int n_res,
                                                              uint64_t* __restrict__ out) {
    batch_resident_block(qp, T, N, n_res, out);
}

// Large batches: kResParts blocks each sum a contiguous range of tokens per
// expert (thread = expert x token quarter, the quarters then added in order),
// and one block adds the partial sums in block order and ranks the experts.
constexpr int kResParts = 32;
__global__ void __launch_bounds__(256) batch_resident_part_kernel(const float* __restrict__ qp, int T, int N,
                                                                  float* __restrict__ part) {
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
    __shared__ float q4[4][kMaxExperts];
    const int e = threadIdx.x & 63, quarter = threadIdx.x >> 6;
    const int t0 = (int)((long long)blockIdx.x * T / kResParts), t1 = (int)((long long)(blockIdx.x + 1) * T / kResParts);
    const int n = t1 - t0, q0 = t0 + quarter * n / 4, q1 = t0 + (quarter + 1) * n / 4;
    float acc = 0.f;
    if (e < N) {
        int t = q0;
        for (; t + 8 <= q1; t += 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = qp[(size_t)(t + u) * N + e];
#pragma unroll
            for (int u = 0; u < 8; ++u) acc += v[u];
        }
        for (; t < q1; ++t) acc += qp[(size_t)t * N + e];
    }
    q4[quarter][e] = acc;
    __syncthreads();
    if (threadIdx.x < kMaxExperts)
        part[blockIdx.x * kMaxExperts + e] = q4[0][e] + q4[1][e] + q4[2][e] + q4[3][e];
}

__global__ void __launch_bounds__(64) batch_resident_final_kernel(const float* __restrict__ part, int N, int n_res,
                                                                  uint64_t* __restrict__ out) {
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
    __shared__ float tot[kMaxExperts];
    __shared__ uint32_t bits[2];
    const int me = threadIdx.x;
    float s = 0.f;
    for (int b = 0; b < kResParts; ++b) s += part[b * kMaxExperts + me];
    tot[me] = s;
    __syncthreads();
    int rank = 0;
    if (me < N)
        for (int j = 0; j < N; ++j) rank += (tot[j] > tot[me] || (tot[j] == tot[me] && j < me)) ? 1 : 0;
    const uint32_t b = __ballot_sync(0xffffffffu, me < N && rank < n_res);
    if ((me & 31) == 0) bits[me >> 5] = b;
    __syncthreads();
    if (me == 0) *out = (uint64_t)bits[0] | ((uint64_t)bits[1] << 32);
}

// ---------------------------------------------------------------------------
// Miss handling, one warp per token (APEX §4.3 Algorithm 1; SPICE LoRE).
// Lane l holds experts l and l + 32.  Every decision is lane-parallel: the
// misses are classified by ballots, the substitutes are the pool members of
// pool rank below the number of substitutions (one pass of independent rank
// comparisons, as in route_select_token), and each final expert is written to
// its slot (its rank by router probability) by the lane that holds it.
__device__ __forceinline__ void select_token(
    int t, const float* __restrict__ router_prob, const int32_t* __restrict__ topk_idx,
    const uint64_t* __restrict__ prefetch_mask, const uint64_t* __restrict__ resident, int policy,
    float gamma, const int32_t* __restrict__ delta_hat, const int32_t* __restrict__ delta_star,
    int N, int k, int renorm, int32_t* __restrict__ final_idx, float* __restrict__ final_gate,
    int32_t* __restrict__ final_kind, uint64_t* __restrict__ fetch_mask,
    int32_t* __restrict__ counters, DevError* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    const uint64_t vm = valid_mask(N);
    const int e0 = lane, e1 = lane + 32;
    const float a0 = e0 < N ? router_prob[(size_t)t * N + e0] : -INFINITY;
    const float a1 = e1 < N ? router_prob[(size_t)t * N + e1] : -INFINITY;
    // the routed set: lane j < k reads slot j
    const int re = lane < k ? topk_idx[(size_t)t * k + lane] : 0;
    const bool bad = __any_sync(0xffffffffu, lane < k && (re < 0 || re >= N));
    if (bad) {
        if (lane == 0) set_error(err, MOE_ERR_DEVICE_INDEX, t);
        return;
    }
    const uint32_t rlo = __reduce_or_sync(0xffffffffu, lane < k && re < 32 ? 1u << re : 0u);
    const uint32_t rhi = __reduce_or_sync(0xffffffffu, lane < k && re >= 32 ? 1u << (re - 32) : 0u);
    const uint64_t routed = (uint64_t)rlo | ((uint64_t)rhi << 32);
    const uint64_t pref = prefetch_mask ? prefetch_mask[t] : ~0ull;
    const uint64_t res = resident ? *resident : ~0ull;
    const uint64_t avail = pref & res & vm;
    const uint64_t missing = routed & ~avail;
    // misses: LoRE below gamma (HYBRID, HETERO), the rest fetched or substituted
    uint64_t lore = 0, fetch = 0, to_sub = 0;
    if (missing) {
        if (policy == MOE_MISS_EXACT) {
            fetch = missing;
        } else if (policy == MOE_MISS_LORE) {
            lore = missing;
        } else if (policy == MOE_MISS_SUBSTITUTE) {
            to_sub = missing;
        } else {
            const bool l0 = ((missing >> e0) & 1) && a0 < gamma;
            const bool l1 = ((missing >> e1) & 1) && a1 < gamma;
            lore = (uint64_t)__ballot_sync(0xffffffffu, l0) | ((uint64_t)__ballot_sync(0xffffffffu, l1) << 32);
            if (policy == MOE_MISS_HETERO) fetch = missing & ~lore;  // exact either way: fetch or host
            else to_sub = missing & ~lore;
        }
    }
    // substitutes: the available, non-routed experts with the largest router
    // probability, one per substituted miss (the whole pool if it is smaller)
    const uint64_t pool = avail & ~routed;
    const int n_sub = __popcll(to_sub);
    uint64_t subs = 0;
    bool shortfall = false;
    if (n_sub > 0) {
        if (__popcll(pool) <= n_sub) {
            subs = pool;
            shortfall = __popcll(pool) < n_sub;
        } else {
            int p0 = 0, p1 = 0;  // pool members ahead of e0 / e1
#pragma unroll 8
            for (int j = 0; j < 64; ++j) {
                const float aj = __shfl_sync(0xffffffffu, j < 32 ? a0 : a1, j & 31);
                const bool in = (pool >> j) & 1;
                p0 += (in && (aj > a0 || (aj == a0 && j < e0))) ? 1 : 0;
                p1 += (in && (aj > a1 || (aj == a1 && j < e1))) ? 1 : 0;
            }
            const bool s0 = ((pool >> e0) & 1) && p0 < n_sub, s1 = ((pool >> e1) & 1) && p1 < n_sub;
            subs = (uint64_t)__ballot_sync(0xffffffffu, s0) | ((uint64_t)__ballot_sync(0xffffffffu, s1) << 32);
        }
    }
    const uint64_t fin = (routed & ~missing) | lore | fetch | subs;
    // canonical slot order: descending router probability, lowest index first
    // (each final expert's rank among the at most k final experts)
    int c0 = 0, c1 = 0;
    for (uint64_t m = fin; m; m &= m - 1) {
        const int j = __ffsll((long long)m) - 1;
        const float aj = __shfl_sync(0xffffffffu, j < 32 ? a0 : a1, j & 31);
        c0 += (aj > a0 || (aj == a0 && j < e0)) ? 1 : 0;
        c1 += (aj > a1 || (aj == a1 && j < e1)) ? 1 : 0;
    }
    const bool f0 = (fin >> e0) & 1, f1 = (fin >> e1) & 1;
    const int nf = __popcll(fin);
    float gsum = 0.f;
    if (renorm) {  // the final gates summed in slot order
        float g = 0.f;
        for (int j = 0; j < nf; ++j) {
            const uint32_t b0 = __ballot_sync(0xffffffffu, f0 && c0 == j);
            const uint32_t b1 = __ballot_sync(0xffffffffu, f1 && c1 == j);
            const int src = b0 ? __ffs(b0) - 1 : __ffs(b1) - 1;
            const float v = __shfl_sync(0xffffffffu, b0 ? a0 : a1, src);
            g += v;
        }
        gsum = g;
    }
    auto put = [&](int slot, int e, float a) {
        const size_t sl = (size_t)t * k + slot;
        final_idx[sl] = e;
        final_gate[sl] = (renorm && gsum > 0.f) ? a / gsum : a;
        final_kind[sl] = ((lore >> e) & 1) ? MOE_KIND_LORE : ((fetch >> e) & 1) ? MOE_KIND_FETCH : MOE_KIND_COMPUTE;
    };
    if (f0 && c0 < k) put(c0, e0, a0);
    if (f1 && c1 < k) put(c1, e1, a1);
    if (lane >= nf && lane < k) {  // fewer final experts than slots (a capacity shortfall)
        const size_t sl = (size_t)t * k + lane;
        final_idx[sl] = -1;
        final_gate[sl] = 0.f;
        final_kind[sl] = MOE_KIND_COMPUTE;
    }
    if (lane == 0) {
        if (fetch_mask && fetch) atomicOr(reinterpret_cast<unsigned long long*>(fetch_mask),
                                          (unsigned long long)fetch);
        if (counters) {
            atomicAdd(&counters[MOE_CNT_HIT], __popcll(routed & avail));
            atomicAdd(&counters[MOE_CNT_SUBSTITUTE], __popcll(subs));
            atomicAdd(&counters[MOE_CNT_LORE], __popcll(lore));
            atomicAdd(&counters[MOE_CNT_FETCH], __popcll(fetch));
            if (prefetch_mask) atomicAdd(&counters[MOE_CNT_OVERLAP], (routed & ~pref) == 0 ? 1 : 0);
            if (delta_hat) atomicAdd(&counters[MOE_CNT_DELTA_HAT], delta_hat[t]);
            if (delta_star) atomicAdd(&counters[MOE_CNT_DELTA_STAR], delta_star[t]);
            if (shortfall) atomicAdd(&counters[MOE_CNT_SHORTFALL], 1);
        }
        if (shortfall) set_error(err, MOE_ERR_CAPACITY, t);
    }
}

__global__ void __launch_bounds__(256) select_resident_kernel(
    const float* __restrict__ router_prob, const int32_t* __restrict__ topk_idx,
    const uint64_t* __restrict__ prefetch_mask, const uint64_t* __restrict__ resident, int policy,
    float gamma, const int32_t* __restrict__ delta_hat, const int32_t* __restrict__ delta_star, int T,
    int N, int k, int renorm, int32_t* __restrict__ final_idx, float* __restrict__ final_gate,
    int32_t* __restrict__ final_kind, uint64_t* __restrict__ fetch_mask,
    int32_t* __restrict__ counters, DevError* __restrict__ err) {
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
    // the block's counters and fetch mask gathered in shared memory, then one
    // global atomic each (every token adding to the same global counters
    // serialised on them)
    __shared__ int32_t s_cnt[MOE_NUM_COUNTERS];
    __shared__ unsigned long long s_fetch;
    if (threadIdx.x < MOE_NUM_COUNTERS) s_cnt[threadIdx.x] = 0;
    if (threadIdx.x == 0) s_fetch = 0ull;
    __syncthreads();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp < T)
        select_token(warp, router_prob, topk_idx, prefetch_mask, resident, policy, gamma, delta_hat, delta_star,
                     N, k, renorm, final_idx, final_gate, final_kind,
                     fetch_mask ? reinterpret_cast<uint64_t*>(&s_fetch) : nullptr, counters ? s_cnt : nullptr,
                     err);
    __syncthreads();
    if (counters && threadIdx.x < MOE_NUM_COUNTERS && s_cnt[threadIdx.x])
        atomicAdd(&counters[threadIdx.x], s_cnt[threadIdx.x]);
    if (fetch_mask && threadIdx.x == 0 && s_fetch)
        atomicOr(reinterpret_cast<unsigned long long*>(fetch_mask), s_fetch);
}

// ---------------------------------------------------------------------------
// Fused front end of a small batch (see launch_route_front).  After the
// logits, the last block keeps every per-token intermediate in shared memory
// (the token-tile staging area, free by then): it loads the logits once,
// runs selection, resident set and miss handling on shared copies, writes the
// outputs out with coalesced stores and permutes from the shared copies.
struct FrontSmem {  // byte offsets into the dynamic shared memory
    int lr, lp, sc, prob, qp, tki, tkg, dh, pm, ds, fi, fg, fk, bres, th, total;
};

__host__ __device__ inline FrontSmem front_smem(int T, int N, int k) {
    FrontSmem f;
    int o = 0;
    auto take = [&](int bytes) { const int at = o; o = (o + bytes + 15) & ~15; return at; };
    f.lr = take(T * N * 4); f.lp = take(T * N * 4); f.sc = take(T * 4); f.prob = take(T * N * 4);
    f.qp = take(T * N * 4); f.tki = take(T * k * 4); f.tkg = take(T * k * 4); f.dh = take(T * 4);
    f.pm = take(T * 8); f.ds = take(T * 4); f.fi = take(T * k * 4); f.fg = take(T * k * 4);
    f.fk = take(T * k * 4); f.bres = take(8); f.th = take(kMaxExperts * 4);  // theta (delta_max + 1 <= N)
    f.total = o;
    return f;
}

template <typename W, int TT>
__global__ void __launch_bounds__(256) route_front_kernel(const __grid_constant__ FrontArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int s_last;
    const LogitsArgs& la = a.la;
    const int n_out = la.has_prefetch ? 2 * la.N + 1 : la.N;
    logits_tile<W, TT>((const W*)la.x, (const W*)(la.x_pre ? la.x_pre : la.x), (const W*)la.w_router, la.bias,
                       (const W*)la.w_prefetch, la.w_ord, la.T, la.d, la.N, n_out, 8, la.logits_r, la.logits_p,
                       la.score, smem_raw);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(a.ticket, 1) == (int)(gridDim.x * gridDim.y) - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    grid_dep_launch();  // the FFN may start its prologue during the per-token stages
    const int tid = threadIdx.x, warp = tid >> 5, nw = blockDim.x >> 5;
    const RouteSelectArgs& ra = a.ra;
    const SelectArgs& sa = a.sa;
    const int T = ra.T, N = ra.N, k = ra.k;
    const FrontSmem F = front_smem(T, N, k);
    float* lr = reinterpret_cast<float*>(smem_raw + F.lr);
    float* lp = reinterpret_cast<float*>(smem_raw + F.lp);
    float* sc = reinterpret_cast<float*>(smem_raw + F.sc);
    float* prob = reinterpret_cast<float*>(smem_raw + F.prob);
    float* qp = reinterpret_cast<float*>(smem_raw + F.qp);
    int32_t* tki = reinterpret_cast<int32_t*>(smem_raw + F.tki);
    float* tkg = reinterpret_cast<float*>(smem_raw + F.tkg);
    int32_t* dh = reinterpret_cast<int32_t*>(smem_raw + F.dh);
    uint64_t* pm = reinterpret_cast<uint64_t*>(smem_raw + F.pm);
    int32_t* ds = reinterpret_cast<int32_t*>(smem_raw + F.ds);
    int32_t* fi = reinterpret_cast<int32_t*>(smem_raw + F.fi);
    float* fg = reinterpret_cast<float*>(smem_raw + F.fg);
    int32_t* fk = reinterpret_cast<int32_t*>(smem_raw + F.fk);
    uint64_t* bres = reinterpret_cast<uint64_t*>(smem_raw + F.bres);
    float* th = reinterpret_cast<float*>(smem_raw + F.th);
    // the other blocks' logits, once (past L1)
    for (int i = tid; i < T * N; i += blockDim.x) {
        lr[i] = __ldcg(ra.logits_r + i);
        if (ra.has_prefetch) lp[i] = __ldcg(ra.logits_p + i);
    }
    if (ra.has_prefetch) {
        for (int i = tid; i < T; i += blockDim.x) sc[i] = __ldcg(ra.score + i);
        for (int i = tid; i <= ra.delta_max; i += blockDim.x) th[i] = ra.theta[i];  // with the logits, not later
    }
    __syncthreads();
    for (int t = warp; t < T; t += nw)
        route_select_token(t, lr, lp, sc, th, ra.logit_tau, N, k, ra.delta_max, ra.has_prefetch, tki, tkg,
                           prob, dh, pm, ra.delta_star ? ds : nullptr, ra.qp ? qp : nullptr);
    __syncthreads();
    for (int i = tid; i < T * N; i += blockDim.x) ra.router_prob[i] = prob[i];
    for (int i = tid; i < T * k; i += blockDim.x) { ra.topk_idx[i] = tki[i]; ra.topk_gate[i] = tkg[i]; }
    for (int i = tid; i < T; i += blockDim.x) {
        ra.delta_hat[i] = dh[i];
        ra.prefetch_mask[i] = pm[i];
        if (ra.delta_star) ra.delta_star[i] = ds[i];
    }
    if (a.n_resident > 0) {
        batch_resident_block(qp, T, N, a.n_resident, bres);
        if (tid == 0) *a.batch_resident = *bres;
    }
    // the slot counters and the fetch mask gather in shared memory and go out
    // with plain stores (this block is their only writer): global atomics on
    // lines this thread has just cleared cost microseconds on the critical path
    __shared__ int32_t s_cnt[MOE_NUM_COUNTERS];
    __shared__ unsigned long long s_fetch;
    if (tid < MOE_NUM_COUNTERS) s_cnt[tid] = 0;
    if (tid == 0) s_fetch = 0ull;
    __syncthreads();
    const uint64_t* resident = a.n_resident > 0 ? bres : sa.resident;
    for (int t = warp; t < T; t += nw)
        select_token(t, prob, tki, sa.prefetch_mask ? pm : nullptr, resident, sa.policy, sa.gamma, dh,
                     sa.delta_star ? ds : nullptr, N, k, sa.renorm, fi, fg, fk,
                     sa.fetch_mask ? reinterpret_cast<uint64_t*>(&s_fetch) : nullptr, sa.counters ? s_cnt : nullptr,
                     sa.err);
    __syncthreads();
    if (sa.counters && tid < MOE_NUM_COUNTERS) sa.counters[tid] = s_cnt[tid];
    if (sa.fetch_mask && tid == 0) *sa.fetch_mask = s_fetch;
    for (int i = tid; i < T * k; i += blockDim.x) {
        sa.final_idx[i] = fi[i];
        sa.final_gate[i] = fg[i];
        sa.final_kind[i] = fk[i];
    }
    const PermuteArgs& pa = a.pa;
    permute_block(fi, fk, pa.n_slots, pa.N, pa.expert_offsets, pa.perm, pa.inv_perm, pa.err, a.plan);
    if (tid == 0) *a.ticket = 0;
}

template <typename W>
static cudaError_t launch_front_t(const FrontArgs& a, cudaStream_t st) {
    constexpr int TT = 8;
    const LogitsArgs& la = a.la;
    const int n_out = la.has_prefetch ? 2 * la.N + 1 : la.N;
    dim3 grid((la.T + TT - 1) / TT, (n_out + 7) / 8);
    const size_t stage = (size_t)2 * TT * la.d * sizeof(W);
    const size_t tail = (size_t)front_smem(la.T, la.N, a.ra.k).total;
    const size_t smem = stage > tail ? stage : tail;
    cudaError_t e = allow_max_smem(route_front_kernel<W, TT>);
    if (e != cudaSuccess) return e;
    route_front_kernel<W, TT><<<grid, 256, smem, st>>>(a);
    return note_launch(reinterpret_cast<const void*>(route_front_kernel<W, TT>), 256, smem, cudaGetLastError());
}

cudaError_t launch_route_front(const FrontArgs& a, cudaStream_t st) {
    if (a.pa.n_slots > kFrontMaxSlots || a.la.T > kFrontMaxTokens) return cudaErrorInvalidValue;
    return a.la.bf16 ? launch_front_t<__nv_bfloat16>(a, st) : launch_front_t<float>(a, st);
}

// ---------------------------------------------------------------------------
// host launchers

template <typename W>
static cudaError_t launch_logits_t(const LogitsArgs& a, cudaStream_t st) {
    constexpr int TT = 8;
    const bool sep_pre = a.x_pre != nullptr && a.x_pre != a.x;
    if (a.part && route_tc_usable(a.T, a.d, a.N, a.bf16, a.has_prefetch, sep_pre)) {
        cudaError_t e = launch_route_tc(a, a.part, st);
        if (e != cudaSuccess || !a.has_prefetch) return e;
        return launch_pdl(route_score_kernel<W>, dim3((a.T + 7) / 8), dim3(256), 0, st,
                          (const W*)(a.x_pre ? a.x_pre : a.x), a.w_ord, a.T, a.d, a.score);
    }
    // (a row quad must not straddle the router / prefetch-router boundary when
    // the two routers read different inputs)
    if (a.T >= 2048 && (a.x_pre == nullptr || a.x_pre == a.x || a.N % 4 == 0)) {
        const int rows = a.has_prefetch ? 2 * a.N : a.N;
        dim3 grid((a.T + 63) / 64, (rows + 63) / 64);
        route_logits_tiled_kernel<W><<<grid, 256, 0, st>>>(
            (const W*)a.x, (const W*)(a.x_pre ? a.x_pre : a.x), (const W*)a.w_router, a.bias,
            (const W*)a.w_prefetch, a.w_ord, a.T, a.d, a.N, rows, a.logits_r, a.logits_p, a.score);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess || !a.has_prefetch) return e;
        return launch_pdl(route_score_kernel<W>, dim3((a.T + 7) / 8), dim3(256), 0, st,
                          (const W*)(a.x_pre ? a.x_pre : a.x), a.w_ord, a.T, a.d, a.score);
    }
    const int n_out = a.has_prefetch ? 2 * a.N + 1 : a.N;
    const int t_tiles = (a.T + TT - 1) / TT;
    const int rows_per_block = 8;
    const int threads = 256;
    dim3 grid(t_tiles, (n_out + rows_per_block - 1) / rows_per_block);
    const size_t smem = (size_t)2 * TT * a.d * sizeof(W);
    if (smem > 48 * 1024) {
        cudaError_t e = allow_max_smem(route_logits_kernel<W, TT>);
        if (e != cudaSuccess) return e;
    }
    route_logits_kernel<W, TT><<<grid, threads, smem, st>>>(
        (const W*)a.x, (const W*)(a.x_pre ? a.x_pre : a.x), (const W*)a.w_router, a.bias,
        (const W*)a.w_prefetch, a.w_ord, a.T, a.d, a.N, n_out, rows_per_block, a.logits_r,
        a.logits_p, a.score);
    return cudaGetLastError();
}

cudaError_t launch_logits(const LogitsArgs& a, cudaStream_t st) {
    return a.bf16 ? launch_logits_t<__nv_bfloat16>(a, st) : launch_logits_t<float>(a, st);
}

cudaError_t launch_route_select(const RouteSelectArgs& a, cudaStream_t st) {
    const int warps = 8;
    dim3 grid((a.T + warps - 1) / warps);
    return launch_pdl(route_select_kernel, grid, dim3(warps * 32), 0, st, a.logits_r, a.logits_p, a.score, a.theta,
                      a.logit_tau, a.T, a.N, a.k, a.delta_max, a.has_prefetch, a.topk_idx, a.topk_gate,
                      a.router_prob, a.delta_hat, a.prefetch_mask, a.delta_star, a.qp);
}

cudaError_t launch_batch_resident(const float* qp, int T, int N, int n_res, uint64_t* out, float* part,
                                  cudaStream_t st) {
    if (T >= 8 * kResParts && part) {
        cudaError_t e = launch_pdl(batch_resident_part_kernel, dim3(kResParts), dim3(256), 0, st, qp, T, N, part);
        if (e != cudaSuccess) return e;
        return launch_pdl(batch_resident_final_kernel, dim3(1), dim3(64), 0, st, (const float*)part, N, n_res, out);
    } else {
        batch_resident_kernel<<<1, 1024, 0, st>>>(qp, T, N, n_res, out);
    }
    return cudaGetLastError();
}

cudaError_t launch_select_resident(const SelectArgs& a, cudaStream_t st) {
    const int warps = 8;
    dim3 grid((a.T + warps - 1) / warps);
    return launch_pdl(select_resident_kernel, grid, dim3(warps * 32), 0, st, a.router_prob, a.topk_idx,
                      a.prefetch_mask, a.resident, a.policy, a.gamma, a.delta_hat, a.delta_star, a.T, a.N, a.k,
                      a.renorm, a.final_idx, a.final_gate, a.final_kind, a.fetch_mask, a.counters, a.err);
}

}  // namespace moe
