// Bit-sliced expert weights: a low-precision draft of the expert FFN.
//
// ELMoE-3D (CSDN post), bit-slicing section: each weight is an INT8 value
// with a scale shared by every precision; its 8 bits are stored as 8 binary
// planes, and a b-bit representation combines the top b planes (plane 7
// carries -128, plane p < 7 carries 2^p; the learned LSB-enhancement scale is
// not used).  Its data-layout note keeps an expert's planes contiguous so that
// the top b planes are one read.  Layout here, per matrix [R, C] (R output
// rows, C inputs, C a multiple of 32):
//   planes [8][R][C/32] uint32: slot s holds plane 7 - s (MSB first), bit i
//          of word w of row r = bit of q[r][32 w + i]; the top b planes are
//          slots 0 .. b-1, the first b * R * C/32 words;
//   scales [R] float32: s_r = max_c |W[r][c]| / 127, q = rint(W / s_r)
//          clamped to +-127 (symmetric per output row; the pages leave the
//          quantiser open).
// Gate and up are [I, d]; the down projection is packed transposed, [d, I],
// so that every matrix is read as row dot products.
//
// A row dot product over bit planes: sum_k v_k q_b[r][k] = sum over the top b
// planes p of w_p * (sum of v_k over the set bits of plane p).  The masked
// sums come from a table built once per block in shared memory: for every
// group of 4 consecutive inputs, the 16 sums of its subsets, so that a 32-bit
// plane word costs 8 table reads.  Table layout [j][v][w] (j the nibble of
// the word, v the 4-bit pattern, w the word), rows of a fixed 128 words
// (inputs <= 4096): an index is the pattern shifted by a constant plus the
// lane's word, the nibble's row a constant offset; lanes reading consecutive
// words hit distinct banks.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kBsThreads = 512;  // 16 warps per block

constexpr int kBsRowShift = 7;                        // table row = 128 words
constexpr size_t kBsTableBytes = (size_t)8 * 16 * (1 << kBsRowShift) * 4;  // 64 KB

__device__ __forceinline__ float bs_load(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float bs_load(const float* p, size_t i) { return p[i]; }

// ---------------------------------------------------------------- pack
// One block per output row: the row's largest magnitude, its scale, then a
// warp per 32-input word: every lane quantises one input and 8 ballots form
// the word of each plane.
template <typename W>
__global__ void __launch_bounds__(256) bitslice_pack_kernel(const W* __restrict__ w, int rows_in, int cols_in,
                                                           int transpose, uint32_t* __restrict__ planes,
                                                           float* __restrict__ scales) {
    grid_dep_wait();
    __shared__ float red[8];
    const int R = transpose ? cols_in : rows_in, C = transpose ? rows_in : cols_in;
    const int r = blockIdx.x, words = C / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    auto at = [&](int c) -> float {
        return transpose ? bs_load(w, (size_t)c * cols_in + r) : bs_load(w, (size_t)r * cols_in + c);
    };
    float mx = 0.f;
    for (int c = threadIdx.x; c < C; c += blockDim.x) mx = fmaxf(mx, fabsf(at(c)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) mx = fmaxf(mx, red[i]);
    const float s = __fdiv_rn(mx, 127.0f);
    if (threadIdx.x == 0) scales[r] = s;
    for (int wd = warp; wd < words; wd += blockDim.x >> 5) {
        int q = 0;
        if (s > 0.f) {
            q = (int)rintf(__fdiv_rn(at(wd * 32 + lane), s));
            q = q > 127 ? 127 : q < -127 ? -127 : q;
        }
        const unsigned byte = (unsigned)(q & 0xff);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const uint32_t word = __ballot_sync(0xffffffffu, (byte >> p) & 1u);
            if (lane == 0) planes[((size_t)(7 - p) * R + r) * words + wd] = word;
        }
    }
}

// ---------------------------------------------------------------- table
// Subset sums of every 4 consecutive values of v[0 .. cols): tbl[j][v][w].
__device__ __forceinline__ void bs_build_table(const float* __restrict__ v, int cols, float* tbl) {
    const int words = cols / 32;
    for (int n = threadIdx.x; n < cols / 4; n += blockDim.x) {
        const int wd = n % words, j = n / words;  // consecutive threads: consecutive words
        const int k0 = wd * 32 + j * 4;
        float e[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) e[i] = v[k0 + i];
        float sum[16];
        sum[0] = 0.f;
#pragma unroll
        for (int m = 1; m < 16; ++m) sum[m] = sum[m & (m - 1)] + e[__ffs(m) - 1];
#pragma unroll
        for (int m = 0; m < 16; ++m) tbl[((j * 16 + m) << kBsRowShift) + wd] = sum[m];
    }
}

// sum over the set bits of one plane word: 8 table reads (tw = the table at
// this lane's word)
__device__ __forceinline__ float bs_word_sum(const float* tw, uint32_t bits) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        a0 += tw[(j * 16 + ((bits >> (4 * j)) & 15u)) << kBsRowShift];
        a1 += tw[((j + 1) * 16 + ((bits >> (4 * j + 4)) & 15u)) << kBsRowShift];
    }
    return a0 + a1;
}

template <int B>
__device__ __forceinline__ float bs_plane_weight(int slot) {
    return slot == 0 ? -128.f : (float)(1 << (7 - slot));
}

// Slot s of token t: a routed slot (s < k) names idx[t][s] with gate[t][s];
// slot k + i is shared expert i, stored as expert N + i, gate 1.
__device__ __forceinline__ int bs_expert(const BitsliceArgs& a, int t, int s) {
    if (s >= a.k) return a.N + (s - a.k);
    const int e = a.idx[(size_t)t * a.k + s];
    return e >= 0 && e < a.N ? e : -1;  // no expert: a zero contribution
}

// ---------------------------------------------------------------- gate / up
// Block (persistent over rows, token t): the table over x_t, then a warp per
// (slot, channel) row of this token: g and u over the top B planes, h =
// SiLU(g) u.  Routed slots naming no expert in 0..N-1 give h = 0.  A warp
// takes two rows per iteration and loads all their plane words (WPL words a
// lane per plane and matrix, d <= 1024 * WPL) before the table reads that
// consume them, so one row's loads are in flight during the other's sums.
template <typename W, int B, int WPL>
__global__ void __launch_bounds__(kBsThreads) bitslice_gateup_kernel(BitsliceArgs a, const W* __restrict__ x) {
    grid_dep_wait();  // x and the routed experts come from the previous launches
    extern __shared__ __align__(16) float bs_tbl[];
    const int t = blockIdx.y, d = a.d, I = a.I, words = d / 32;
    // the down launch's completion counters start from zero every call
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < a.T * (d / 16); i += blockDim.x) a.cnt[i] = 0;
    float* xv = bs_tbl + kBsTableBytes / 4;  // x_t as float
    for (int i = threadIdx.x; i < d; i += blockDim.x) xv[i] = bs_load(x, (size_t)t * d + i);
    __syncthreads();
    bs_build_table(xv, d, bs_tbl);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const size_t mat = (size_t)8 * I * words;  // words of one expert's matrix
    const int S = a.k + a.ns, rows = S * I, stride = gridDim.x * nw;
    for (int row0 = blockIdx.x * nw + warp; row0 < rows; row0 += 2 * stride) {
        uint32_t bg[2][WPL][B], bu[2][WPL][B];
        int e[2], c[2], slot[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int row = row0 + r * stride;
            slot[r] = row / I;
            c[r] = row % I;
            e[r] = row < rows ? bs_expert(a, t, slot[r]) : -1;
            const bool ok = e[r] >= 0 && e[r] < a.N + a.ns;
            const uint32_t* pg = a.planes_gate + (size_t)(ok ? e[r] : 0) * mat + (size_t)c[r] * words;
            const uint32_t* pu = a.planes_up + (size_t)(ok ? e[r] : 0) * mat + (size_t)c[r] * words;
#pragma unroll
            for (int i = 0; i < WPL; ++i) {
                const int wd = lane + 32 * i;
#pragma unroll
                for (int sl = 0; sl < B; ++sl) {
                    bg[r][i][sl] = ok && wd < words ? pg[(size_t)sl * I * words + wd] : 0u;
                    bu[r][i][sl] = ok && wd < words ? pu[(size_t)sl * I * words + wd] : 0u;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int row = row0 + r * stride;
            if (row >= rows) break;
            float h = 0.f;
            if (e[r] >= 0 && e[r] < a.N + a.ns) {
                float ag = 0.f, au = 0.f;
#pragma unroll
                for (int i = 0; i < WPL; ++i) {
                    const int wd = lane + 32 * i;
                    if (wd < words) {
#pragma unroll
                        for (int sl = 0; sl < B; ++sl) {
                            ag += bs_plane_weight<B>(sl) * bs_word_sum(bs_tbl + wd, bg[r][i][sl]);
                            au += bs_plane_weight<B>(sl) * bs_word_sum(bs_tbl + wd, bu[r][i][sl]);
                        }
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    ag += __shfl_xor_sync(0xffffffffu, ag, o);
                    au += __shfl_xor_sync(0xffffffffu, au, o);
                }
                const float g = ag * a.scales_gate[(size_t)e[r] * I + c[r]];
                const float u = au * a.scales_up[(size_t)e[r] * I + c[r]];
                h = g / (1.f + expf(-g)) * u;
            }
            if (lane == 0) a.h[((size_t)t * S + slot[r]) * I + c[r]] = h;
        }
    }
}

// the y_part rows of one (token, slot) pair: a warp per output j of this
// block's share, two outputs per iteration with all their plane words loaded
// first (WPL words a lane per plane, I <= 1024 * WPL)
template <int B, int WPL>
__device__ __forceinline__ void bs_down_rows(const BitsliceArgs& a, int pair, int e, int lane, int warp, int nw,
                                             float* bs_tbl) {
    const int d = a.d, I = a.I, words = I / 32;
    bs_build_table(a.h + (size_t)pair * I, I, bs_tbl);
    __syncthreads();
    const size_t mat = (size_t)8 * d * words;
    const int stride = gridDim.x * nw;
    for (int j0 = blockIdx.x * nw + warp; j0 < d; j0 += 2 * stride) {
        uint32_t bd[2][WPL][B];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int j = j0 + r * stride;
            const uint32_t* pd = a.planes_down + (size_t)e * mat + (size_t)(j < d ? j : 0) * words;
#pragma unroll
            for (int i = 0; i < WPL; ++i) {
                const int wd = lane + 32 * i;
#pragma unroll
                for (int sl = 0; sl < B; ++sl)
                    bd[r][i][sl] = j < d && wd < words ? pd[(size_t)sl * d * words + wd] : 0u;
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int j = j0 + r * stride;
            if (j >= d) break;
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < WPL; ++i) {
                const int wd = lane + 32 * i;
                if (wd < words) {
#pragma unroll
                    for (int sl = 0; sl < B; ++sl)
                        acc += bs_plane_weight<B>(sl) * bs_word_sum(bs_tbl + wd, bd[r][i][sl]);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) a.y_part[(size_t)pair * d + j] = acc * a.scales_down[(size_t)e * d + j];
        }
    }
}

// ---------------------------------------------------------------- down
// Block (persistent over output rows, (token, slot) pair): the table over
// h of the pair, then a warp per output j: y_part = s_d[j] * the dot of h
// with the top B planes of row j of W_down^T.  Block x of every pair of a
// token covers the same outputs j; the last of them to finish (a counter per
// token and block x) forms y for those outputs: the gated sum over the
// slots in order.
template <int B, int WPL>
__global__ void __launch_bounds__(kBsThreads) bitslice_down_kernel(BitsliceArgs a) {
    grid_dep_wait();  // h and the zeroed counters come from the gate / up launch
    extern __shared__ __align__(16) float bs_tbl[];
    __shared__ int s_last;
    const int pair = blockIdx.y, d = a.d;
    const int S = a.k + a.ns;
    const int t = pair / S;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int e = bs_expert(a, t, pair % S);
    if (e < 0 || e >= a.N + a.ns) {  // no expert: a zero contribution
        for (int j = blockIdx.x * nw + warp; j < d; j += gridDim.x * nw)
            if (lane == 0) a.y_part[(size_t)pair * d + j] = 0.f;
    } else {
        bs_down_rows<B, WPL>(a, pair, e, lane, warp, nw, bs_tbl);
    }
    // the gated sum over the token's slots, by the last block of this x
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(a.cnt + (size_t)t * (d / 16) + blockIdx.x, 1) == S - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int i = threadIdx.x;; i += blockDim.x) {
        const int j = blockIdx.x * nw + (i % nw) + (i / nw) * gridDim.x * nw;
        if (j >= d) break;
        const size_t at = (size_t)t * d + j;
        float acc = a.accumulate ? a.y[at] : 0.f;
        for (int s = 0; s < S; ++s) {
            const float g = (s < a.k && a.gate) ? a.gate[(size_t)t * a.k + s] : 1.f;
            acc += g * __ldcg(a.y_part + ((size_t)t * S + s) * d + j);
        }
        a.y[at] = acc;
    }
}


// ---------------------------------------------------------------- host
cudaError_t launch_bitslice_pack(int rows_in, int cols_in, bool bf16, const void* w, int transpose, uint32_t* planes,
                                 float* scales, cudaStream_t st) {
    const int R = transpose ? cols_in : rows_in;
    if (bf16)
        return launch_pdl(bitslice_pack_kernel<__nv_bfloat16>, dim3(R), dim3(256), 0, st,
                          static_cast<const __nv_bfloat16*>(w), rows_in, cols_in, transpose, planes, scales);
    return launch_pdl(bitslice_pack_kernel<float>, dim3(R), dim3(256), 0, st, static_cast<const float*>(w), rows_in,
                      cols_in, transpose, planes, scales);
}

template <typename W, int B, int WPL1, int WPL2>
static cudaError_t bs_ffn(const BitsliceArgs& a, const void* x, int sms, cudaStream_t st) {
    const size_t smem1 = kBsTableBytes + (size_t)a.d * 4;
    cudaError_t e = allow_max_smem(bitslice_gateup_kernel<W, B, WPL1>);
    if (e != cudaSuccess) return e;
    // gate / up: about two blocks per SM over all tokens
    const int rows1 = (a.k + a.ns) * a.I, per1 = (rows1 + 15) / 16;
    int g1 = (2 * sms + a.T - 1) / a.T;
    g1 = g1 < 1 ? 1 : g1 > per1 ? per1 : g1;
    e = launch_pdl(bitslice_gateup_kernel<W, B, WPL1>, dim3(g1, a.T), dim3(kBsThreads), smem1, st, a,
                   static_cast<const W*>(x));
    if (e != cudaSuccess) return e;
    const size_t smem2 = kBsTableBytes;
    e = allow_max_smem(bitslice_down_kernel<B, WPL2>);
    if (e != cudaSuccess) return e;
    const int pairs = a.T * (a.k + a.ns), per2 = (a.d + 15) / 16;
    int g2 = (2 * sms + pairs - 1) / pairs;
    g2 = g2 < 1 ? 1 : g2 > per2 ? per2 : g2;
    return launch_pdl(bitslice_down_kernel<B, WPL2>, dim3(g2, pairs), dim3(kBsThreads), smem2, st, a);
}

// words a lane per plane: d (gate / up) and I (down) up to 2048 take 2, up to 4096 take 4
template <typename W, int B>
static cudaError_t bs_ffn_w(const BitsliceArgs& a, const void* x, int sms, cudaStream_t st) {
    const bool small1 = a.d <= 2048, small2 = a.I <= 2048;
    if (small1 && small2) return bs_ffn<W, B, 2, 2>(a, x, sms, st);
    if (small1) return bs_ffn<W, B, 2, 4>(a, x, sms, st);
    if (small2) return bs_ffn<W, B, 4, 2>(a, x, sms, st);
    return bs_ffn<W, B, 4, 4>(a, x, sms, st);
}

template <typename W>
static cudaError_t bs_ffn_bits(const BitsliceArgs& a, const void* x, int sms, cudaStream_t st) {
    switch (a.bits) {
        case 1: return bs_ffn_w<W, 1>(a, x, sms, st);
        case 2: return bs_ffn_w<W, 2>(a, x, sms, st);
        case 3: return bs_ffn_w<W, 3>(a, x, sms, st);
        case 4: return bs_ffn_w<W, 4>(a, x, sms, st);
        case 5: return bs_ffn_w<W, 5>(a, x, sms, st);
        case 6: return bs_ffn_w<W, 6>(a, x, sms, st);
        case 7: return bs_ffn_w<W, 7>(a, x, sms, st);
        case 8: return bs_ffn_w<W, 8>(a, x, sms, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bitslice_ffn(const BitsliceArgs& a, const void* x, bool bf16, int sms, cudaStream_t st) {
    return bf16 ? bs_ffn_bits<__nv_bfloat16>(a, x, sms, st) : bs_ffn_bits<float>(a, x, sms, st);
}

size_t bitslice_table_bytes(int) { return kBsTableBytes; }

}  // namespace moe
