// Stage 1 for large batches: the router and prefetch-router logits on the
// 5th-generation tensor cores.
//
// APEX §4.1: the router l = x W_r^T (+ b) and the prefetch router
// l_p = x_pre W_p^T are linear maps of the token state.  With x_pre = x they
// are one GEMM [T, d] x [d, 2N]: the N router rows and the N prefetch rows
// form one B operand of 2N rows.  tcgen05.mma kind::f16 (bf16 operands, fp32
// accumulators in tensor memory), operands brought by TMA into 128-byte
// swizzled shared memory.  Tile = 128 tokens x 2N outputs; d is split over S
// CTAs per tile (S chosen so that the tiles times S cover the SMs), each
// writing an fp32 partial row block; route_tc_reduce_kernel adds the partials
// in split order plus the router bias.  The ordinal scorer w . x_pre (fp32
// weights) stays on route_score_kernel.
//
// Block: 4 warps.  Warp 0 lane 0 issues the TMA loads (ring of kRtStages),
// warp 1 allocates tensor memory and its lane 0 issues the MMAs, then all
// four warps drain the accumulator (thread = tensor-memory lane = token).
// Every wait is bounded; a timeout records MOE_ERR_TIMEOUT and the roles
// leave their loops.
#include <cuda.h>

#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tma.h"

namespace moe {

constexpr int kRtBM = 128, kRtStages = 4, kRtThreads = 128, kRtMaxSplits = 8;
constexpr uint32_t kRtStageA = kRtBM * kTcBK * 2;  // 16 KB

struct RouteTcParams {
    CUtensorMap map_x;   // x [T, d], boxes of 64 values x 128 tokens
    CUtensorMap map_wr;  // w_router [N, d], boxes of 64 values x N rows
    CUtensorMap map_wp;  // w_prefetch [N, d] (n_out = 2N)
    int T, d, N, n_out;  // n_out: the MMA's N (2N, or N without a prefetch router)
    float* part;         // [splits][T][n_out] fp32 partial logits
    DevError* err;
};

__host__ __device__ inline uint32_t rt_stage_bytes(int n_out) {
    return kRtStageA + (((uint32_t)n_out * 128u + 1023u) & ~1023u);
}

__global__ void __launch_bounds__(kRtThreads, 1) route_tc_kernel(const __grid_constant__ RouteTcParams p) {
    grid_dep_wait();  // x is written before this launch; no tensor memory taken before it
    extern __shared__ unsigned char rt_smem_raw[];
    __shared__ __align__(8) uint64_t full[kRtStages], empty[kRtStages], done;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t smem_base = (smem_u32(rt_smem_raw) + 1023u) & ~1023u;
    const uint32_t stage_bytes = rt_stage_bytes(p.n_out);
    const uint32_t tx_bytes = kRtStageA + (uint32_t)p.n_out * 128u;
    const uint32_t tmem_cols = p.n_out <= 32 ? 32 : p.n_out <= 64 ? 64 : p.n_out <= 128 ? 128 : 256;
    volatile int* abort_flag = &abort_s;
    const int m0 = blockIdx.x * kRtBM, split = blockIdx.y, splits = gridDim.y;
    const int nkb = p.d / (int)kTcBK;
    const int kb_begin = split * nkb / splits, kb_end = (split + 1) * nkb / splits;

    if (tid == 0) {
        for (int s = 0; s < kRtStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        fence_mbar_init();
        abort_s = 0;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tmem_base_s)), "r"(tmem_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_s;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        int it = 0;
        for (int kb = kb_begin; kb < kb_end && !*abort_flag; ++kb, ++it) {
            const int st = it % kRtStages;
            if (!tc_wait(&empty[st], ((it / kRtStages) & 1) ^ 1, abort_flag, p.err, 11)) break;
            const uint32_t a_dst = smem_base + st * stage_bytes;
            const uint32_t b_dst = a_dst + kRtStageA;
            mbar_arrive_expect_tx(&full[st], tx_bytes);
            tma_load_2d(a_dst, &p.map_x, kb * kTcBK, m0, &full[st]);
            tma_load_2d(b_dst, &p.map_wr, kb * kTcBK, 0, &full[st]);
            if (p.n_out > p.N) tma_load_2d(b_dst + p.N * 128, &p.map_wp, kb * kTcBK, 0, &full[st]);
        }
        // the loads in flight finish before the block may exit
        for (int k = (it > kRtStages ? it - kRtStages : 0); k < it; ++k)
            (void)tc_wait(&full[k % kRtStages], (k / kRtStages) & 1, abort_flag, p.err, 12, false);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        const uint32_t idesc = tc_idesc(kRtBM, p.n_out, 0);
        int it = 0;
        for (int kb = kb_begin; kb < kb_end; ++kb, ++it) {
            const int st = it % kRtStages;
            if (!tc_wait(&full[st], (it / kRtStages) & 1, abort_flag, p.err, 13)) break;
            tc_fence_after();
            const uint32_t a_addr = smem_base + st * stage_bytes;
            const uint32_t b_addr = a_addr + kRtStageA;
#pragma unroll
            for (int kk = 0; kk < (int)kTcBK / 16; ++kk)
                tc_mma(tmem_base, smem_desc(a_addr + kk * 32, 16, 1024), smem_desc(b_addr + kk * 32, 16, 1024),
                       idesc, (it | kk) ? 1u : 0u);
            tc_commit(&empty[st]);  // frees the stage when these MMAs are done
        }
        tc_commit(&done);  // every MMA issued so far has finished
    }
    __syncwarp();

    // ---------------- epilogue: thread = tensor-memory lane = token m0 + tid
    bool ok = true;
    if (lane == 0) ok = tc_wait(&done, 0, abort_flag, p.err, 14, false) && !*abort_flag;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    tc_fence_after();
    if (ok && kb_end > kb_begin) {
        const int tok = m0 + tid;
        const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16);
        float* dst = p.part + ((size_t)split * p.T + tok) * p.n_out;
        for (int c = 0; c < p.n_out; c += 16) {
            float v[16];
            tmem_ld16(taddr + c, v);
            if (tok < p.T) {
#pragma unroll
                for (int i = 0; i < 16; i += 4)
                    *reinterpret_cast<float4*>(dst + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
            }
        }
    } else if (kb_end <= kb_begin && m0 + tid < p.T) {
        // an empty share of d (more splits than 64-value blocks): zero partial
        float* dst = p.part + ((size_t)split * p.T + m0 + tid) * p.n_out;
        for (int c = 0; c < p.n_out; c += 4) *reinterpret_cast<float4*>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(tmem_cols));
}

// logits = the partials added in split order (+ the router bias); router
// columns to logits_r, prefetch columns to logits_p.  One thread per 4 outputs.
__global__ void __launch_bounds__(256) route_tc_reduce_kernel(const float* __restrict__ part, int splits, int T,
                                                              int N, int n_out, const float* __restrict__ bias,
                                                              float* __restrict__ logits_r,
                                                              float* __restrict__ logits_p) {
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
    const int n4 = n_out / 4;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T * n4; i += gridDim.x * blockDim.x) {
        const int tok = i / n4, c = (i % n4) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < splits; ++s)
            add4(acc, *reinterpret_cast<const float4*>(part + ((size_t)s * T + tok) * n_out + c));
        const float a[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int o = c + j;
            if (o < N) logits_r[(size_t)tok * N + o] = a[j] + (bias ? bias[o] : 0.f);
            else logits_p[(size_t)tok * N + (o - N)] = a[j];
        }
    }
}

bool route_tc_usable(int T, int d, int N, bool bf16, bool has_prefetch, bool sep_pre) {
    if (!bf16 || T <= kTcMinTokens || d % (int)kTcBK != 0 || sep_pre) return false;
    const int n_out = has_prefetch ? 2 * N : N;
    return N % 8 == 0 && n_out % 16 == 0 && n_out >= 16 && n_out <= 256;
}

size_t route_tc_part_bytes(int T, int N) { return (size_t)kRtMaxSplits * T * 2 * N * sizeof(float); }

cudaError_t launch_route_tc(const LogitsArgs& a, float* part, cudaStream_t st) {
    RouteTcParams p;
    std::memset(&p, 0, sizeof(p));
    p.T = a.T; p.d = a.d; p.N = a.N; p.n_out = a.has_prefetch ? 2 * a.N : a.N;
    p.part = part;
    p.err = a.err;
    if (encode_bf16_2d(&p.map_x, a.x, a.d, a.T, (uint64_t)a.d * 2, kTcBK, kRtBM) != MOE_OK ||
        encode_bf16_2d(&p.map_wr, a.w_router, a.d, a.N, (uint64_t)a.d * 2, kTcBK, a.N) != MOE_OK)
        return cudaErrorInvalidValue;
    if (a.has_prefetch &&
        encode_bf16_2d(&p.map_wp, a.w_prefetch, a.d, a.N, (uint64_t)a.d * 2, kTcBK, a.N) != MOE_OK)
        return cudaErrorInvalidValue;
    const int m_tiles = (a.T + kRtBM - 1) / kRtBM, nkb = a.d / (int)kTcBK;
    int splits = (a.sms > 0 ? a.sms : 148) / m_tiles;
    splits = splits < 1 ? 1 : splits > kRtMaxSplits ? kRtMaxSplits : splits;
    if (splits > nkb) splits = nkb;
    const size_t smem = (size_t)kRtStages * rt_stage_bytes(p.n_out) + 1024;
    cudaError_t e = allow_max_smem(route_tc_kernel);
    if (e != cudaSuccess) return e;
    e = note_launch(reinterpret_cast<const void*>(route_tc_kernel), kRtThreads, smem,
                    launch_pdl(route_tc_kernel, dim3(m_tiles, splits), dim3(kRtThreads), smem, st, p));
    if (e != cudaSuccess) return e;
    const int n4 = a.T * (p.n_out / 4);
    const int blocks = (n4 + 255) / 256 < 4 * 152 ? (n4 + 255) / 256 : 4 * 152;
    return launch_pdl(route_tc_reduce_kernel, dim3(blocks), dim3(256), 0, st, (const float*)part, splits, a.T, a.N,
                      p.n_out, a.bias, a.logits_r, a.logits_p);
}

}  // namespace moe
