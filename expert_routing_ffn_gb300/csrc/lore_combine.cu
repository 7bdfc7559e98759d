// Stages 4 and 5: the SPICE LoRE surrogate residual and the combine.
//
// SPICE write-up, LoRE section: a missing expert e is approximated by
// y_shared + B_e A_e h with A_e [r, d], B_e [d, r], r << d; the shared part
// is added once per token by the combine, scaled by the LoRE slots' gates.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "mma_sync.cuh"

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

// ---------------------------------------------------------------------------
// Large batches: the LoRE slots grouped by expert (launch_group_lore), so that
// A_e and B_e are read once per tile of up to kLoreTile slots of e instead of
// once per slot.  Tile index -> (expert, first grouped position) from the
// per-expert tile counts; every block walks tiles blockIdx.x, + gridDim.x, ...
// These two kernels are the CUDA-core forms (fp32 layers, other ranks):
// register-tiled, operands staged in shared memory K-major as fp32, thread =
// 4 x 4 outputs from two 16-byte shared loads per step.  bf16 layers with r a
// multiple of 16 up to 64 take the warp-level MMA forms below.
constexpr int kLoreTile = 64;
constexpr int kLoreKC = 32;  // values of d per shared-memory chunk (z pass)
constexpr int kLoreKS = 8;   // d split over this many blocks per tile (z pass)

// the expert and first grouped position of tile `tile`; false past the last tile
__device__ __forceinline__ bool lore_tile_of(const int* s_off, int N, int tile, int& e, int& first) {
    int t0 = 0;
    for (int x = 0; x < N; ++x) {
        const int n = (s_off[x + 1] - s_off[x] + kLoreTile - 1) / kLoreTile;
        if (tile < t0 + n) { e = x; first = s_off[x] + (tile - t0) * kLoreTile; return true; }
        t0 += n;
    }
    return false;
}

__device__ __forceinline__ void fma4x4(float (&acc)[4][4], const float4& a, const float4& b) {
    const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        fma2(acc[i][0], acc[i][1], av[i], av[i], b.x, b.y);
        fma2(acc[i][2], acc[i][3], av[i], av[i], b.z, b.w);
    }
}

// zp[ks, pos, q] = A_e[q, d-range ks] . x_t[d-range ks] for the slots of a
// tile (pos = grouped position): d is split over kLoreKS blocks (blockIdx.y),
// whose partials lore_b_grouped_kernel adds in ks order.  Thread (slot quad
// sq, rank quad rq), 4 r threads computing; d in chunks of kLoreKC, the next
// chunk's global loads in flight during the current one.
template <typename W>
__global__ void __launch_bounds__(256) lore_z_grouped_kernel(const W* __restrict__ x,
                                                             const W* __restrict__ A,
                                                             const int32_t* __restrict__ g_off,
                                                             const int32_t* __restrict__ g_list, int d, int k,
                                                             int r, int N, int n_pos, float* __restrict__ zp) {
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
    constexpr int V = Vec<W>::n;
    constexpr int CV = kLoreKC / V;                    // 16-byte vectors per row and chunk
    constexpr int XL = (kLoreTile * CV + 255) / 256;   // x vectors per thread and chunk
    constexpr int AL = (64 * CV + 255) / 256;          // A vectors per thread and chunk (r <= 64)
    __shared__ __align__(16) float xs[kLoreKC][kLoreTile];
    __shared__ __align__(16) float as[kLoreKC][64];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_tok[kLoreTile];
    const int tid = threadIdx.x, sq = tid & 15, rq = tid >> 4;
    const bool computes = rq * 4 < r;
    for (int i = tid; i <= N; i += blockDim.x) s_off[i] = g_off[i];
    __syncthreads();
    int e, first;
    for (int tile = blockIdx.x; lore_tile_of(s_off, N, tile, e, first); tile += gridDim.x) {
        const int nt = min(kLoreTile, s_off[e + 1] - first);
        if (tid < kLoreTile) s_tok[tid] = tid < nt ? g_list[first + tid] / k : -1;
        __syncthreads();
        const W* Ae = A + (size_t)e * r * d;
        uint4 rx[XL], ra[AL];
        auto load = [&](int k0) {
#pragma unroll
            for (int j = 0; j < XL; ++j) {
                const int i = tid + 256 * j, row = i % kLoreTile, cv = i / kLoreTile;
                rx[j] = make_uint4(0, 0, 0, 0);
                if (cv < CV && s_tok[row] >= 0 && k0 + cv * V < d)
                    rx[j] = *reinterpret_cast<const uint4*>(x + (size_t)s_tok[row] * d + k0 + cv * V);
            }
#pragma unroll
            for (int j = 0; j < AL; ++j) {
                const int i = tid + 256 * j, q = i % 64, cv = i / 64;
                ra[j] = make_uint4(0, 0, 0, 0);
                if (cv < CV && q < r && k0 + cv * V < d)
                    ra[j] = *reinterpret_cast<const uint4*>(Ae + (size_t)q * d + k0 + cv * V);
            }
        };
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        const int n_chunks = (d + kLoreKC - 1) / kLoreKC, ks = blockIdx.y;
        const int k_begin = ks * n_chunks / kLoreKS * kLoreKC;
        const int k_end = min(d, (ks + 1) * n_chunks / kLoreKS * kLoreKC);
        if (k_begin < k_end) load(k_begin);
        for (int k0 = k_begin; k0 < k_end; k0 += kLoreKC) {
#pragma unroll
            for (int j = 0; j < XL; ++j) {
                const int i = tid + 256 * j, row = i % kLoreTile, cv = i / kLoreTile;
                if (cv < CV) {
                    float v[V];
                    unpack16(rx[j], v, (W*)nullptr);
#pragma unroll
                    for (int u = 0; u < V; ++u) xs[cv * V + u][row] = v[u];
                }
            }
#pragma unroll
            for (int j = 0; j < AL; ++j) {
                const int i = tid + 256 * j, q = i % 64, cv = i / 64;
                if (cv < CV) {
                    float v[V];
                    unpack16(ra[j], v, (W*)nullptr);
#pragma unroll
                    for (int u = 0; u < V; ++u) as[cv * V + u][q] = v[u];
                }
            }
            __syncthreads();
            if (k0 + kLoreKC < k_end) load(k0 + kLoreKC);
            if (computes) {
                const int kc = min(kLoreKC, d - k0);
                if (kc == kLoreKC) {
#pragma unroll
                    for (int kk = 0; kk < kLoreKC; ++kk)
                        fma4x4(acc, *reinterpret_cast<const float4*>(&xs[kk][sq * 4]),
                               *reinterpret_cast<const float4*>(&as[kk][rq * 4]));
                } else {
                    for (int kk = 0; kk < kc; ++kk)
                        fma4x4(acc, *reinterpret_cast<const float4*>(&xs[kk][sq * 4]),
                               *reinterpret_cast<const float4*>(&as[kk][rq * 4]));
                }
            }
            __syncthreads();
        }
        if (computes) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int p = sq * 4 + i;
                if (p >= nt) continue;
                *reinterpret_cast<float4*>(zp + ((size_t)ks * n_pos + first + p) * r + rq * 4) =
                    make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            }
        }
        __syncthreads();  // s_tok is rewritten by the next tile
    }
}

// zg[pos, :] = g_slot * (the kLoreKS partials zp[., pos, :] added in order),
// for the n = g_off[N] grouped positions; one thread per 4 rank values.
__global__ void __launch_bounds__(256) lore_z_sum_kernel(const float* __restrict__ final_gate,
                                                         const int32_t* __restrict__ g_off,
                                                         const int32_t* __restrict__ g_list, int r, int N,
                                                         int n_pos, const float* __restrict__ zp,
                                                         float* __restrict__ zg) {
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
    const int n = g_off[N];
    const int r4 = r / 4;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n * r4; i += gridDim.x * blockDim.x) {
        const int pos = i / r4, q4 = i % r4;
        float4 p[kLoreKS];
#pragma unroll
        for (int ks = 0; ks < kLoreKS; ++ks)
            p[ks] = *reinterpret_cast<const float4*>(zp + ((size_t)ks * n_pos + pos) * r + q4 * 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int ks = 0; ks < kLoreKS; ++ks) add4(acc, p[ks]);
        const float g = final_gate[g_list[pos]];
        *reinterpret_cast<float4*>(zg + (size_t)pos * r + q4 * 4) =
            make_float4(g * acc.x, g * acc.y, g * acc.z, g * acc.w);
    }
}

// v[pos, c] = B_e[c, :] . zg[pos] for the slots of a tile (pos = grouped
// position) and the columns c of this block's share of d (blockIdx.y of
// kLoreBY shares, in chunks of 64 columns, the next chunk's B_e rows in flight
// during the current one).  Thread (slot quad, column quad).
constexpr int kLoreBY = 4;
template <typename W>
__global__ void __launch_bounds__(256) lore_b_grouped_kernel(const W* __restrict__ B,
                                                             const int32_t* __restrict__ g_off, int d, int r,
                                                             int N, const float* __restrict__ zg,
                                                             float* __restrict__ v) {
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
    constexpr int V = Vec<W>::n;
    constexpr int TC = 64;                 // columns per chunk
    constexpr int BL = (64 * TC / V + 255) / 256;  // B vectors per thread and chunk (r <= 64)
    __shared__ __align__(16) float zs[64][kLoreTile];  // [q][slot]
    __shared__ __align__(16) float bs[64][TC];         // [q][column]
    __shared__ int s_off[kMaxExperts + 1];
    const int tid = threadIdx.x, sq = tid & 15, cq = tid >> 4;
    const int n_chunks = (d + TC - 1) / TC;
    const int ch_begin = blockIdx.y * n_chunks / kLoreBY, ch_end = (blockIdx.y + 1) * n_chunks / kLoreBY;
    const int rv = r / V;  // r * sizeof(W) is a multiple of 16 on this path
    for (int i = tid; i <= N; i += blockDim.x) s_off[i] = g_off[i];
    __syncthreads();
    int e, first;
    for (int tile = blockIdx.x; lore_tile_of(s_off, N, tile, e, first); tile += gridDim.x) {
        const int nt = min(kLoreTile, s_off[e + 1] - first);
        // z rows: 64 x r / 4 float4, two per thread at r = 32
        for (int i0 = tid; i0 < kLoreTile * r / 4; i0 += 2 * blockDim.x) {
            float4 zz[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * blockDim.x, row = i % kLoreTile;
                zz[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < kLoreTile * r / 4 && row < nt)
                    zz[u] = *reinterpret_cast<const float4*>(zg + (size_t)(first + row) * r + (i / kLoreTile) * 4);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * blockDim.x, row = i % kLoreTile, q4 = i / kLoreTile;
                if (i < kLoreTile * r / 4) {
                    zs[q4 * 4 + 0][row] = zz[u].x; zs[q4 * 4 + 1][row] = zz[u].y;
                    zs[q4 * 4 + 2][row] = zz[u].z; zs[q4 * 4 + 3][row] = zz[u].w;
                }
            }
        }
        const W* Be = B + (size_t)e * d * r;
        uint4 rb[BL];
        auto load = [&](int ch) {
#pragma unroll
            for (int j = 0; j < BL; ++j) {
                const int i = tid + 256 * j, col = i % TC, qv = i / TC, c = ch * TC + col;
                rb[j] = make_uint4(0, 0, 0, 0);
                if (qv < rv && c < d) rb[j] = *reinterpret_cast<const uint4*>(Be + (size_t)c * r + qv * V);
            }
        };
        if (ch_begin < ch_end) load(ch_begin);
        for (int ch = ch_begin; ch < ch_end; ++ch) {
            __syncthreads();  // bs free (previous chunk), zs written (first chunk)
#pragma unroll
            for (int j = 0; j < BL; ++j) {
                const int i = tid + 256 * j, col = i % TC, qv = i / TC;
                if (qv < rv) {
                    float b[V];
                    unpack16(rb[j], b, (W*)nullptr);
#pragma unroll
                    for (int u = 0; u < V; ++u) bs[qv * V + u][col] = b[u];
                }
            }
            __syncthreads();
            if (ch + 1 < ch_end) load(ch + 1);
            float acc[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;
            for (int q = 0; q < r; ++q)
                fma4x4(acc, *reinterpret_cast<const float4*>(&zs[q][sq * 4]),
                       *reinterpret_cast<const float4*>(&bs[q][cq * 4]));
            const int col = ch * TC + cq * 4;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (sq * 4 + i >= nt || col >= d) continue;
                *reinterpret_cast<float4*>(v + (size_t)(first + sq * 4 + i) * d + col) =
                    make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            }
        }
        __syncthreads();  // zs is rewritten by the next tile
    }
}

// ---------------------------------------------------------------------------
// The same two products for bf16 layers on the tensor cores, as warp-level
// MMAs with register operands (mma.sync): the rank r (16 to 64) is too short
// a side for a shared-memory-staged tcgen05 tile, and with fragments loaded
// straight from global memory no staging or block barrier is needed.  A warp
// works on 16 grouped positions of one expert (kLoreMT), rows g = lane / 4
// and g + 8 of each fragment, tq = lane % 4 the thread within its group.
// Within a K step the products may be summed in any order, so each thread
// loads contiguous 16-byte pieces and assigns their elements to the
// fragment's K slots by a fixed bijection (the same on both operands).
constexpr int kLoreMT = 16;     // grouped positions per warp tile
constexpr int kLoreCB = 256;    // columns of d per warp item (B pass)

// the expert and first grouped position of 16-position tile `tile` (tile
// prefix counts in s_toff); false past the last tile
__device__ __forceinline__ bool lore_mtile_of(const int* s_off, const int* s_toff, int N, int tile, int& e,
                                              int& first) {
    if (tile >= s_toff[N]) return false;
    int lo = 0, hi = N - 1;  // the last expert with s_toff[e] <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_toff[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    e = lo;
    first = s_off[e] + (tile - s_toff[e]) * kLoreMT;
    return true;
}

// s_off = g_off, s_toff[e] = 16-position tiles of the experts before e
// (warp 0 scans: lane l holds experts l and l + 32)
__device__ __forceinline__ void lore_mtile_table(const int32_t* __restrict__ g_off, int N, int* s_off,
                                                 int* s_toff) {
    for (int i = threadIdx.x; i <= N; i += blockDim.x) s_off[i] = g_off[i];
    __syncthreads();
    if (threadIdx.x < 32) {
        // exclusive prefix in expert order: experts 0..31 (lane l: c0), then
        // 32..63 (lane l: c1), each half an inclusive warp scan
        const int l = threadIdx.x;
        const int c0 = l < N ? (s_off[l + 1] - s_off[l] + kLoreMT - 1) / kLoreMT : 0;
        const int c1 = l + 32 < N ? (s_off[l + 33] - s_off[l + 32] + kLoreMT - 1) / kLoreMT : 0;
        int a = c0, b = c1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ta = __shfl_up_sync(0xffffffffu, a, o), tb = __shfl_up_sync(0xffffffffu, b, o);
            if (l >= o) { a += ta; b += tb; }
        }
        const int half = __shfl_sync(0xffffffffu, a, 31), rest = __shfl_sync(0xffffffffu, b, 31);
        if (l < N) s_toff[l] = a - c0;
        if (l + 32 < N) s_toff[l + 32] = half + b - c1;
        if (l == 0) s_toff[N] = half + rest;
    }
    __syncthreads();
}

// zp[ks, pos, :] = A_e x_t over the d-range ks (of kLoreKS) for a 16-position
// tile: M = positions, N = the R rank rows (R / 8 MMA columns), K = d in steps
// of 32 values.  Thread tq's 16-byte piece [8 tq, 8 tq + 8) of a 32-value
// step holds K slots {2tq, 2tq+1 | 2tq+8, 2tq+9} of two 16-deep MMA steps:
// elements (0,1 | 2,3) for the first, (4,5 | 6,7) for the second.
template <int R>
__global__ void __launch_bounds__(256) lore_z_mma_kernel(const __nv_bfloat16* __restrict__ x,
                                                         const __nv_bfloat16* __restrict__ A,
                                                         const int32_t* __restrict__ g_off,
                                                         const int32_t* __restrict__ g_list, int d, int k, int N,
                                                         int n_pos, float* __restrict__ zp) {
    grid_dep_wait();  // the grouping comes from the previous kernels
    __shared__ int s_off[kMaxExperts + 1], s_toff[kMaxExperts + 1];
    lore_mtile_table(g_off, N, s_off, s_toff);
    const int lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
    const int warps = gridDim.x * (blockDim.x >> 5);
    const int kc = d / kLoreKS;  // values of d per split (a multiple of 32)
    const int items = s_toff[N] * kLoreKS;
    for (int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < items; item += warps) {
        const int tile = item / kLoreKS, ks = item % kLoreKS;
        int e, first;
        if (!lore_mtile_of(s_off, s_toff, N, tile, e, first)) break;
        const int nt = min(kLoreMT, s_off[e + 1] - first);
        const int t0 = g < nt ? g_list[first + g] / k : -1;
        const int t1 = g + 8 < nt ? g_list[first + g + 8] / k : -1;
        const uint4* x0 = t0 >= 0 ? reinterpret_cast<const uint4*>(x + (size_t)t0 * d) : nullptr;
        const uint4* x1 = t1 >= 0 ? reinterpret_cast<const uint4*>(x + (size_t)t1 * d) : nullptr;
        const uint4* a_rows = reinterpret_cast<const uint4*>(A + ((size_t)e * R + g) * d);  // row 8j + g: + 8j*d
        float acc[R / 8][4];
#pragma unroll
        for (int j = 0; j < R / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        const int v_lo = (ks * kc) / 8 + tq, v_hi = ((ks + 1) * kc) / 8;  // 16-byte vector indices
#pragma unroll 2
        for (int v = v_lo; v < v_hi; v += 4) {
            const uint4 p0 = x0 ? __ldg(x0 + v) : make_uint4(0, 0, 0, 0);
            const uint4 p1 = x1 ? __ldg(x1 + v) : make_uint4(0, 0, 0, 0);
            uint4 bw[R / 8];
#pragma unroll
            for (int j = 0; j < R / 8; ++j) bw[j] = __ldg(a_rows + (size_t)j * d + v);
#pragma unroll
            for (int j = 0; j < R / 8; ++j) {
                mma_bf16_16816(acc[j], p0.x, p1.x, p0.y, p1.y, bw[j].x, bw[j].y);
                mma_bf16_16816(acc[j], p0.z, p1.z, p0.w, p1.w, bw[j].z, bw[j].w);
            }
        }
#pragma unroll
        for (int j = 0; j < R / 8; ++j) {
            const int q = 8 * j + 2 * tq;
            if (g < nt)
                *reinterpret_cast<float2*>(zp + ((size_t)ks * n_pos + first + g) * R + q) =
                    make_float2(acc[j][0], acc[j][1]);
            if (g + 8 < nt)
                *reinterpret_cast<float2*>(zp + ((size_t)ks * n_pos + first + g + 8) * R + q) =
                    make_float2(acc[j][2], acc[j][3]);
        }
    }
}

// v[pos, c] = B_e[c, :] . zg[pos] for a 16-position tile and kLoreCB columns:
// M = positions, N = columns (8 per MMA), K = R in tf32 steps of 8 (zg is
// fp32; B_e's bf16 values are exact in tf32).  Thread tq's pair [2tq, 2tq+2)
// of an 8-value step holds K slots tq and tq + 4.  The zg fragments are
// loaded once per item and held across the columns.
template <int R>
__global__ void __launch_bounds__(256) lore_b_mma_kernel(const __nv_bfloat16* __restrict__ B,
                                                         const int32_t* __restrict__ g_off, int d, int N,
                                                         const float* __restrict__ zg, float* __restrict__ v) {
    grid_dep_wait();  // zg comes from the previous kernel
    __shared__ int s_off[kMaxExperts + 1], s_toff[kMaxExperts + 1];
    lore_mtile_table(g_off, N, s_off, s_toff);
    const int lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
    const int warps = gridDim.x * (blockDim.x >> 5);
    const int n_cb = d / kLoreCB;
    const int items = s_toff[N] * n_cb;
    for (int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < items; item += warps) {
        const int tile = item / n_cb, cb = item % n_cb;
        int e, first;
        if (!lore_mtile_of(s_off, s_toff, N, tile, e, first)) break;
        const int nt = min(kLoreMT, s_off[e + 1] - first);
        uint32_t af[R / 8][4];
#pragma unroll
        for (int s = 0; s < R / 8; ++s) {
            float2 z0 = make_float2(0.f, 0.f), z1 = make_float2(0.f, 0.f);
            if (g < nt) z0 = *reinterpret_cast<const float2*>(zg + (size_t)(first + g) * R + 8 * s + 2 * tq);
            if (g + 8 < nt) z1 = *reinterpret_cast<const float2*>(zg + (size_t)(first + g + 8) * R + 8 * s + 2 * tq);
            af[s][0] = to_tf32(z0.x); af[s][1] = to_tf32(z1.x);
            af[s][2] = to_tf32(z0.y); af[s][3] = to_tf32(z1.y);
        }
        const __nv_bfloat16* Be = B + (size_t)e * d * R;
        const int c_begin = cb * kLoreCB;
#pragma unroll 4
        for (int c0 = c_begin; c0 < c_begin + kLoreCB; c0 += 8) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t* brow = reinterpret_cast<const uint32_t*>(Be + (size_t)(c0 + g) * R) + tq;
#pragma unroll
            for (int s = 0; s < R / 8; ++s) {
                const uint32_t w = __ldg(brow + 4 * s);  // B_e[c0 + g][8s + 2tq, + 1]
                mma_tf32_1688(acc, af[s][0], af[s][1], af[s][2], af[s][3], w << 16, w & 0xffff0000u);
            }
            const int c = c0 + 2 * tq;
            if (g < nt) *reinterpret_cast<float2*>(v + (size_t)(first + g) * d + c) = make_float2(acc[0], acc[1]);
            if (g + 8 < nt)
                *reinterpret_cast<float2*>(v + (size_t)(first + g + 8) * d + c) = make_float2(acc[2], acc[3]);
        }
    }
}

// y_lore[t] = the token's LoRE rows v[pos], added in slot order from zero.
__global__ void __launch_bounds__(256) lore_sum_kernel(const int32_t* __restrict__ g_pos, const float* __restrict__ v,
                                                       int d, int k, float* __restrict__ y_lore) {
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
    const int t = blockIdx.x;
    const int q = blockIdx.y * blockDim.x + threadIdx.x;  // float4 column group
    __shared__ int s_pos[kMaxTopK];
    if (threadIdx.x < k) s_pos[threadIdx.x] = g_pos[(size_t)t * k + threadIdx.x];
    __syncthreads();
    if (q >= d / 4) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < k; ++s)
        if (s_pos[s] >= 0) add4(acc, reinterpret_cast<const float4*>(v + (size_t)s_pos[s] * d)[q]);
    reinterpret_cast<float4*>(y_lore + (size_t)t * d)[q] = acc;
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
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
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

// moe_layer_forward's tail on the tensor-core prefill path: combine_kernel
// with the LoRE term summed here from the slots' B_e z rows (v, grouped
// positions) instead of a y_lore row written by a separate launch.  The
// operations are those of lore_sum_kernel then combine_kernel, element by
// element, so the result is bitwise that of the stage-wise calls.
__global__ void __launch_bounds__(256) prefill_epilogue_kernel(const PrefillEpilogueArgs a) {
    grid_dep_wait();  // the FFN's y rows and the LoRE rows (dependent launch)
    const int t = blockIdx.x;
    const int q = blockIdx.y * blockDim.x + threadIdx.x;  // float4 column group
    const int k = a.k, d = a.d;
    __shared__ int s_pos[kMaxTopK], s_lp[kMaxTopK], s_kind[kMaxTopK];
    __shared__ float s_g[kMaxTopK];
    __shared__ float s_lg;
    if (threadIdx.x < k) {  // one thread per slot
        const size_t sl = (size_t)t * k + threadIdx.x;
        s_pos[threadIdx.x] = a.inv_perm[sl];
        s_g[threadIdx.x] = a.final_gate[sl];
        s_kind[threadIdx.x] = a.final_kind[sl];
        s_lp[threadIdx.x] = a.lore_v ? a.g_pos[sl] : -1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // the LoRE gates summed in slot order
        float lg = 0.f;
        for (int s = 0; s < k; ++s)
            if (s_kind[s] == MOE_KIND_LORE) lg += s_g[s];
        s_lg = lg;
    }
    __syncthreads();
    if (q >= d / 4) return;
    const float sh_scale = 1.f + s_lg;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.y_shared) {
        const float4 v = reinterpret_cast<const float4*>(a.y_shared + (size_t)t * d)[q];
        acc.x = v.x * sh_scale; acc.y = v.y * sh_scale; acc.z = v.z * sh_scale; acc.w = v.w * sh_scale;
    }
    for (int s = 0; s < k; ++s) {
        const int pos = s_pos[s];
        if (pos < 0) continue;
        const float g = s_g[s];
        const float4 v = reinterpret_cast<const float4*>(a.y_perm + (size_t)pos * d)[q];
        acc.x = fmaf(g, v.x, acc.x); acc.y = fmaf(g, v.y, acc.y);
        acc.z = fmaf(g, v.z, acc.z); acc.w = fmaf(g, v.w, acc.w);
    }
    if (a.lore_v) {
        float4 yl = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < k; ++s)
            if (s_lp[s] >= 0) add4(yl, reinterpret_cast<const float4*>(a.lore_v + (size_t)s_lp[s] * d)[q]);
        acc.x += yl.x; acc.y += yl.y; acc.z += yl.z; acc.w += yl.w;
    }
    reinterpret_cast<float4*>(a.out + (size_t)t * d)[q] = acc;
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
//
// The slots, the permutation and the plan were written before the expert FFN
// started (the FFN's own wait on them returned before it let this launch
// begin), so they are read, and the LoRE B rows prefetched into L2, before
// the wait on the FFN; its partial rows and the LoRE z rows after it.
template <typename W, bool DIRECT>
__global__ void __launch_bounds__(DIRECT ? 256 : 1024) layer_epilogue_kernel(const EpilogueArgs a) {
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
    if (warp == lore_warp && a.lore_b && col_ok) {
        // this lane's four B rows of each LoRE slot: 4 r contiguous values
        const char* B = static_cast<const char*>(a.lore_b);
        for (int i = 0; i < s_nl; ++i) {
            const int e = s_e[s_lore[i]];
            const char* p = B + ((size_t)e * d + (size_t)q * 4) * r * sizeof(W);
            for (int off = 0; off < 4 * r * (int)sizeof(W); off += 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(p + off));
        }
    }
    grid_dep_wait();  // the FFN's partial rows (and, through the join, LoRE z)
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

template <typename W>
static cudaError_t launch_lore_grouped(const LoreArgs& a, cudaStream_t st) {
    PermuteArgs pa;
    pa.final_idx = a.final_idx; pa.final_kind = a.final_kind; pa.n_slots = a.T * a.k; pa.N = a.N;
    pa.expert_offsets = a.g_off; pa.perm = a.g_list; pa.inv_perm = a.g_pos; pa.err = a.err;
    cudaError_t e = launch_group_lore(pa, a.g_counts, st);
    if (e != cudaSuccess) return e;
    // tiles: at most T*k / kLoreTile + N
    const int n_pos = a.T * a.k;
    const int tiles = n_pos / kLoreTile + a.N;
    const int gz = tiles < 160 ? tiles : 160;
    // bf16, r in {16, 32, 48, 64}, d a multiple of 256: the MMA forms
    const bool mma = std::is_same<W, __nv_bfloat16>::value && a.r % 16 == 0 && a.r >= 16 && a.r <= 64 &&
                     a.d % (kLoreKS * 32) == 0 && a.d % kLoreCB == 0;
    const int mtiles = n_pos / kLoreMT + a.N;  // 16-position tiles, at most
    const int g_cap = 4 * 152;
    if (mma) {
        const int gzm = std::min(g_cap, (mtiles * kLoreKS + 7) / 8);
        const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(a.x);
        const __nv_bfloat16* Ab = static_cast<const __nv_bfloat16*>(a.A);
        auto zk = a.r == 16 ? lore_z_mma_kernel<16> : a.r == 32 ? lore_z_mma_kernel<32>
                : a.r == 48 ? lore_z_mma_kernel<48> : lore_z_mma_kernel<64>;
        e = launch_pdl(zk, dim3(gzm), dim3(256), 0, st, xb, Ab, (const int32_t*)a.g_off,
                       (const int32_t*)a.g_list, a.d, a.k, a.N, n_pos, a.zp);
    } else {
        e = launch_pdl(lore_z_grouped_kernel<W>, dim3(gz, kLoreKS), dim3(256), 0, st, (const W*)a.x, (const W*)a.A,
                       (const int32_t*)a.g_off, (const int32_t*)a.g_list, a.d, a.k, a.r, a.N, n_pos, a.zp);
    }
    if (e != cudaSuccess) return e;
    e = launch_pdl(lore_z_sum_kernel, dim3(4 * 152), dim3(256), 0, st, a.final_gate, (const int32_t*)a.g_off,
                   (const int32_t*)a.g_list, a.r, a.N, n_pos, (const float*)a.zp, a.z);
    if (e != cudaSuccess) return e;
    if (mma) {
        const int gbm = std::min(g_cap, (mtiles * (a.d / kLoreCB) + 7) / 8);
        const __nv_bfloat16* Bb = static_cast<const __nv_bfloat16*>(a.B);
        auto bk = a.r == 16 ? lore_b_mma_kernel<16> : a.r == 32 ? lore_b_mma_kernel<32>
                : a.r == 48 ? lore_b_mma_kernel<48> : lore_b_mma_kernel<64>;
        e = launch_pdl(bk, dim3(gbm), dim3(256), 0, st, Bb, (const int32_t*)a.g_off, a.d, a.N,
                       (const float*)a.z, a.v);
    } else {
        const int gx = tiles < 304 ? tiles : 304;
        e = launch_pdl(lore_b_grouped_kernel<W>, dim3(gx, kLoreBY), dim3(256), 0, st, (const W*)a.B,
                       (const int32_t*)a.g_off, a.d, a.r, a.N, (const float*)a.z, a.v);
    }
    if (e != cudaSuccess || a.skip_sum) return e;
    return launch_pdl(lore_sum_kernel, dim3(a.T, (a.d / 4 + 255) / 256), dim3(256), 0, st, (const int32_t*)a.g_pos,
                      (const float*)a.v, a.d, a.k, a.y_lore);
}

bool lore_grouped_usable(int T, int d, int r, bool bf16) {
    const int esize = bf16 ? 2 : 4;
    return T > kTcMinTokens && r <= 64 && (r * esize) % 16 == 0 && d % 4 == 0 && (d * esize) % 16 == 0;
}

cudaError_t launch_lore(const LoreArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    if (a.v && lore_grouped_usable(a.T, a.d, a.r, a.bf16))
        return a.bf16 ? launch_lore_grouped<__nv_bfloat16>(a, st) : launch_lore_grouped<float>(a, st);
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

cudaError_t launch_prefill_epilogue(const PrefillEpilogueArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    return launch_pdl(prefill_epilogue_kernel, dim3(a.T, (a.d / 4 + 255) / 256), dim3(256), 0, st, a);
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    dim3 grid(a.T, (a.d / 4 + 255) / 256);
    return launch_pdl(combine_kernel, grid, dim3(256), 0, st, a.y_perm, a.inv_perm, a.final_gate, a.final_kind,
                      a.y_shared, a.y_lore, a.d, a.k, a.out);
}

}  // namespace moe
