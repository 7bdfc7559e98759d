// Stage 3b, decode-size batches on the tensor cores.
//
// With a handful of tokens per expert the expert FFN streams weight bytes,
// but a CUDA-core GEMV over several token rows spends a few instructions per
// weight byte (bf16 unpacking, one FMA per row and element, cross-lane sums)
// and becomes issue-bound.  Here the contraction goes to tcgen05 with the
// weights on the M side and the token rows on the N side:
//   gate/up:  G[c, t] = sum_k Wg[c, k] x[t, k],  U likewise
//             (M = 128 channels, N = NT token rows, K = d; A = weight rows,
//             K-major; B = token rows, K-major)
//   h[c, t] = SiLU(G[c, t]) U[c, t]   (epilogue: tensor memory -> bf16 in
//             shared memory, laid out as the next MMA's B operand)
//   down:     Y[j, t] = sum_c Wd[c, j] h[c, t]
//             (M = 128 columns of d, N = NT, K = channels; A = Wd, MN-major;
//             B = h, K-major)
// (FloE method §1 with the identity mask.)  One thread issues a few MMAs per
// 32 KB of weights; the other warps only move accumulators.
//
// Work split: the GEMV plan (segments = an expert with up to NT token rows;
// the channels of all segments concatenated and cut into G equal ranges that
// are multiples of 16, one per CTA).  A CTA's piece of a segment is processed
// in chunks of up to kHT x 128 channels: phase A streams the chunk's gate and
// up rows (64 values of k per stage) and leaves h in shared memory; phase B
// streams the chunk's Wd rows (128 columns of d per stage group) and writes
// Y for those columns into the CTA's partial rows of the segment (later
// chunks add to them).  The GEMV's reduction kernel then sums the partial
// rows of each output row in a fixed order.
//
// Token rows: a shared-expert segment's rows are consecutive tokens of x (one
// box of NT rows); a routed segment's rows of a batch of up to 16 tokens are
// loaded straight from x, one 128-byte box per token (its tokens looked up in
// perm once), those of larger batches from a gathered copy x_perm (one box).
//
// Block: warp 0 issues the TMA loads (ring of kNS stages), warp 1 allocates
// tensor memory and issues the MMAs, warps 2-5 run the epilogues (thread =
// tensor-memory lane = channel in phase A, column of d in phase B).  Every
// wait is bounded; a timeout records MOE_ERR_TIMEOUT and all roles leave.
#include <cuda.h>

#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tma.h"

namespace moe {

constexpr int kTcdThreads = 192;
constexpr uint32_t kTcdW = 128 * 128;  // one matrix per stage: 128 rows x 128 bytes (16 KB)

template <int NT>
struct TcdCfg {
    static constexpr uint32_t kX = NT * 128;             // token tile: NT rows x 64 values
    static constexpr uint32_t kStage = 2 * kTcdW + kX;    // A: gate, up, tokens; B: Wd (2 halves)
    static constexpr int kHT = 4;                         // 128-channel tiles per chunk
    static constexpr uint32_t kHTile = NT * 256;          // h tile: NT rows x 128 channels (bf16)
    static constexpr uint32_t kH = kHT * kHTile;
    static constexpr int kNS = (int)((210u * 1024u - kH) / kStage);
    static constexpr uint32_t kSmem = kNS * kStage + kH + 1024;  // + alignment slack
    static constexpr uint32_t kTmemCols = NT == 16 ? 128 : 256;
    static_assert(kStage % 1024 == 0 && kHTile % 1024 == 0, "1024-byte aligned swizzle atoms");
    static_assert(kNS >= 2, "pipeline depth");
    static_assert(6 * NT <= (int)kTmemCols, "accumulators fit the allocation");
};

struct TcdParams {
    CUtensorMap map_x;   // x [T, d], box {64, NT}: shared-expert segments (rows = tokens t0 ..)
    CUtensorMap map_x1;  // x [T, d], box {64, 1}:  routed segments, one token row per box (NT = 16)
    CUtensorMap map_xp;  // x_perm [T*k, d], box {64, NT}: routed segments, gathered rows (NT = 32)
    const int32_t* perm;  // permuted position -> slot t * k + s
    int topk;
    const ExpertEntry* table;
    const PlanHeader* hdr;
    const Seg* segs;
    float* partial;
    float* u_out;  // up-only mode: u[pos, channel] (fp32, row = permuted position, I columns)
    int d, N, I;
    DevError* err;
    int n_prefetch;  // shared experts to pull into L2 before the dependent-launch wait
};

// One CTA's pieces of segments, as every role walks them.
struct TcdWalk {
    const Seg* segs;
    int n_seg, seg, ch, hi;
    __device__ bool next(Seg& S, int& llo, int& lhi) {
        if (ch >= hi || seg >= n_seg) return false;
        S = segs[seg];
        llo = ch - S.ch_start;
        lhi = min(hi, S.ch_start + S.I) - S.ch_start;
        ch = S.ch_start + lhi;
        ++seg;
        return true;
    }
};

__device__ __forceinline__ bool tcd_begin(const TcdParams& p, TcdWalk& w) {
    const PlanHeader hdr = *p.hdr;
    const int cta = blockIdx.x;
    if (cta >= hdr.G || hdr.n_seg <= 0) return false;
    const int lo = cta * hdr.P, hi = min(lo + hdr.P, hdr.total_ch);
    if (lo >= hi) return false;
    int s_lo = 0, s_hi = hdr.n_seg - 1;
    while (s_lo < s_hi) {
        const int mid = (s_lo + s_hi + 1) >> 1;
        if (p.segs[mid].ch_start <= lo) s_lo = mid; else s_hi = mid - 1;
    }
    w.segs = p.segs; w.n_seg = hdr.n_seg; w.seg = s_lo; w.ch = lo; w.hi = hi;
    return true;
}

// UP = true: FloE's first pass, U = W_up x only (phase A without gate, no
// phase B), written to p.u_out for every routed row and channel of the plan.
template <int NT, bool UP>
__global__ void __launch_bounds__(kTcdThreads, 1) ffn_tcd_kernel(const __grid_constant__ TcdParams p) {
    using C = TcdCfg<NT>;
    constexpr int NS = C::kNS, HT = C::kHT;
    extern __shared__ unsigned char tcd_smem_raw[];
    __shared__ __align__(8) uint64_t full[NS], empty[NS], afull[2], aempty[2], yfull[2], yempty[2],
        hready[HT], drain;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t smem_base = (smem_u32(tcd_smem_raw) + 1023u) & ~1023u;
    const uint32_t h_base = smem_base + NS * C::kStage;
    volatile int* abort_flag = &abort_s;
    const int d = p.d;
    const int nkA = d / 64, nkB = d / 128;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&afull[b], 1);
            mbar_init(&aempty[b], 4);  // one arrival per epilogue warp
            mbar_init(&yfull[b], 1);
            mbar_init(&yempty[b], 4);
        }
        for (int t = 0; t < HT; ++t) mbar_init(&hready[t], 4);
        mbar_init(&drain, 1);
        fence_mbar_init();
        abort_s = 0;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tmem_base_s)), "r"(C::kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_s;
    // tensor-memory columns: G/U of phase-A buffer b at b*2NT (+NT), Y buffer b at 4NT + b*NT
    if (warp == 0 && p.n_prefetch > 0)
        l2_prefetch_shared_experts(p.table, p.N, p.n_prefetch, d, 2, blockIdx.x, gridDim.x, lane);
    grid_dep_wait();  // the plan, perm and x come from the previous kernels
    TcdWalk walk;
    const bool has_work = tcd_begin(p, walk);

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0 && has_work) {
            const uint64_t pol_w = l2_evict_first_policy();
            int it = 0;
            Seg S;
            int llo, lhi;
            bool ok = true;
            auto acquire = [&](uint32_t bytes) -> int {
                const int st = it % NS;
                if (!tc_wait(&empty[st], ((it / NS) & 1) ^ 1, abort_flag, p.err, 11)) return -1;
                mbar_arrive_expect_tx(&full[st], bytes);
                return st;
            };
            int tok[NT];  // routed segment: the token of each row
            while (ok && walk.next(S, llo, lhi)) {
                const ExpertEntry* E = p.table + S.expert;
                const bool shared = S.expert >= p.N;
                // routed rows of up to 16 tokens: one box per row straight from x; of 32:
                // one box from the gathered copy
                const bool per_row = !shared && NT == 16;
                if (per_row)
                    for (int i = 0; i < S.rows && i < NT; ++i) tok[i] = p.perm[S.row0 + i] / p.topk;
                const uint32_t xbytes = per_row ? (uint32_t)min(S.rows, NT) * 128u : C::kX;
                for (int c0 = llo; ok && c0 < lhi; c0 += HT * 128) {
                    const int clen = min(HT * 128, lhi - c0);
                    const int ntl = (clen + 127) / 128;
                    // phase A: gate and up rows of every tile, 64 values of k per stage
                    for (int t = 0; ok && t < ntl; ++t) {
                        const int rows = min(128, clen - t * 128);
                        for (int kc = 0; kc < nkA; ++kc, ++it) {
                            const int st = acquire((UP ? 1u : 2u) * rows * 128u + xbytes);
                            if (st < 0) { ok = false; break; }
                            const uint32_t dst = smem_base + st * C::kStage;
                            if (rows == 128) {  // whole tile: one 128-row box per matrix
                                if (!UP)
                                    tma_load_2d_hint(dst, E->tmap[0], kc * 64, c0 + t * 128, &full[st], pol_w);
                                tma_load_2d_hint(dst + kTcdW, E->tmap[1], kc * 64, c0 + t * 128, &full[st], pol_w);
                            } else {
                                for (int j = 0; j < rows / 16; ++j) {
                                    if (!UP)
                                        tma_load_2d_hint(dst + j * 2048, E->tmap_dec[0], kc * 64,
                                                         c0 + t * 128 + j * 16, &full[st], pol_w);
                                    tma_load_2d_hint(dst + kTcdW + j * 2048, E->tmap_dec[1], kc * 64,
                                                     c0 + t * 128 + j * 16, &full[st], pol_w);
                                }
                            }
                            if (per_row) {
                                for (int i = 0; i < S.rows && i < NT; ++i)
                                    tma_load_2d(dst + 2 * kTcdW + i * 128, &p.map_x1, kc * 64, tok[i], &full[st]);
                            } else {
                                tma_load_2d(dst + 2 * kTcdW, shared ? &p.map_x : &p.map_xp, kc * 64, S.row0,
                                            &full[st]);
                            }
                        }
                    }
                    // phase B: Wd rows of every tile, 128 columns of d per stage
                    for (int dc = 0; !UP && ok && dc < nkB; ++dc) {
                        for (int t = 0; t < ntl; ++t, ++it) {
                            const int rows = min(128, clen - t * 128);
                            const int st = acquire(2u * rows * 128u);
                            if (st < 0) { ok = false; break; }
                            const uint32_t dst = smem_base + st * C::kStage;
                            // whole 64-row blocks with the 64-row down map, the rest in 16-row boxes
                            const int r64 = rows & ~63;
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                for (int q = 0; q < r64; q += 64)
                                    tma_load_2d_hint(dst + hf * kTcdW + q * 128, E->tmap[2], dc * 128 + hf * 64,
                                                     c0 + t * 128 + q, &full[st], pol_w);
                                for (int q = r64; q < rows; q += 16)
                                    tma_load_2d_hint(dst + hf * kTcdW + q * 128, E->tmap_dec[2],
                                                     dc * 128 + hf * 64, c0 + t * 128 + q, &full[st], pol_w);
                            }
                        }
                    }
                }
            }
            grid_dep_launch();  // every load issued: the next kernel may start its prologue
            // wait for the last loads in flight before the block may exit
            for (int k = (it > NS ? it - NS : 0); k < it; ++k)
                (void)tc_wait(&full[k % NS], (k / NS) & 1, abort_flag, p.err, 12, false);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0 && has_work) {
            constexpr uint32_t idA = tc_idesc(128, NT, 0, 0);
            constexpr uint32_t idB = tc_idesc(128, NT, 0, 1);
            int it = 0, na = 0, ny = 0;
            int hph[HT];
#pragma unroll
            for (int t = 0; t < HT; ++t) hph[t] = 0;
            Seg S;
            int llo, lhi;
            bool ok = true;
            while (ok && walk.next(S, llo, lhi)) {
                for (int c0 = llo; ok && c0 < lhi; c0 += HT * 128) {
                    const int clen = min(HT * 128, lhi - c0);
                    const int ntl = (clen + 127) / 128;
                    for (int t = 0; ok && t < ntl; ++t, ++na) {
                        const int ab = na & 1;
                        if (!tc_wait(&aempty[ab], ((na >> 1) & 1) ^ 1, abort_flag, p.err, 13)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t tg = tmem_base + ab * 2 * NT, tu = tg + NT;
                        for (int kc = 0; kc < nkA; ++kc, ++it) {
                            const int st = it % NS;
                            if (!tc_wait(&full[st], (it / NS) & 1, abort_flag, p.err, 14)) { ok = false; break; }
                            tc_fence_after();
                            const uint32_t a = smem_base + st * C::kStage;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint64_t bx = smem_desc(a + 2 * kTcdW + kk * 32, 16, 1024);
                                const uint32_t acc = (kc | kk) ? 1u : 0u;
                                if (!UP) tc_mma(tg, smem_desc(a + kk * 32, 16, 1024), bx, idA, acc);
                                tc_mma(tu, smem_desc(a + kTcdW + kk * 32, 16, 1024), bx, idA, acc);
                            }
                            tc_commit(&empty[st]);
                        }
                        if (!ok) break;
                        tc_commit(&afull[ab]);
                    }
                    if constexpr (!UP) {
                        // every h tile of the chunk written by the epilogue
                        for (int t = 0; ok && t < ntl; ++t) {
                            if (!tc_wait(&hready[t], hph[t] & 1, abort_flag, p.err, 15)) ok = false;
                            ++hph[t];
                        }
                        tc_fence_after();
                        for (int dc = 0; ok && dc < nkB; ++dc, ++ny) {
                            const int yb = ny & 1;
                            if (!tc_wait(&yempty[yb], ((ny >> 1) & 1) ^ 1, abort_flag, p.err, 16)) { ok = false; break; }
                            tc_fence_after();
                            const uint32_t ty = tmem_base + 4 * NT + yb * NT;
                            for (int t = 0; t < ntl; ++t, ++it) {
                                const int rows = min(128, clen - t * 128);
                                const int st = it % NS;
                                if (!tc_wait(&full[st], (it / NS) & 1, abort_flag, p.err, 17)) { ok = false; break; }
                                tc_fence_after();
                                const uint32_t a = smem_base + st * C::kStage;
                                const uint32_t hb = h_base + t * C::kHTile;
                                for (int j = 0; j < rows / 16; ++j) {
                                    const uint64_t ad = smem_desc(a + j * 2048, kTcdW, 1024);
                                    const uint64_t bd = smem_desc(hb + (j >> 2) * (NT * 128) + (j & 3) * 32, 16, 1024);
                                    tc_mma(ty, ad, bd, idB, (t | j) ? 1u : 0u);
                                }
                                tc_commit(&empty[st]);
                            }
                            if (!ok) break;
                            tc_commit(&yfull[yb]);
                        }
                    }
                }
            }
            // every MMA this thread issued has finished before tensor memory is released
            tc_commit(&drain);
            (void)tc_wait(&drain, 0, abort_flag, p.err, 18, false);
        }
    } else if (has_work) {
        // ---------------- epilogue: warps 2..5, thread = tensor-memory lane
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        int na = 0, ny = 0;
        Seg S;
        int llo, lhi;
        bool ok = true;
        auto wait_warp = [&](uint64_t* bar, uint32_t par, int where) -> bool {
            bool w = true;
            if (lane == 0) w = tc_wait(bar, par, abort_flag, p.err, where);
            return __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
        };
        while (ok && walk.next(S, llo, lhi)) {
            const int R = S.rows;
            float* prow = p.partial + (size_t)(S.pbase + (blockIdx.x - S.c0) * S.rows) * d;
            for (int c0 = llo, chunk = 0; ok && c0 < lhi; c0 += HT * 128, ++chunk) {
                const int clen = min(HT * 128, lhi - c0);
                const int ntl = (clen + 127) / 128;
                // phase A epilogues: h = SiLU(G) U for this thread's channel
                for (int t = 0; t < ntl; ++t, ++na) {
                    const int ab = na & 1;
                    if (!wait_warp(&afull[ab], (na >> 1) & 1, 19)) { ok = false; break; }
                    tc_fence_after();
                    const int rows = min(128, clen - t * 128);
                    const uint32_t tg = tmem_base + lane_off + ab * 2 * NT;
                    if (UP) {
                        // u[row0 + tok, channel] for this thread's channel
                        const int ch = c0 + t * 128 + r;
#pragma unroll 1
                        for (int c = 0; c < NT && c < R; c += 16) {
                            float u[16];
                            tmem_ld16(tg + NT + c, u);
                            if (r < rows) {
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    if (c + i < R) p.u_out[(size_t)(S.row0 + c + i) * p.I + ch] = u[i];
                            }
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&aempty[ab]);
                        continue;
                    }
                    unsigned char* hb = tcd_smem_raw + (h_base - smem_u32(tcd_smem_raw)) + t * C::kHTile +
                                        (r >> 6) * (NT * 128);
                    const int cin = r & 63;
#pragma unroll 1
                    for (int c = 0; c < NT && c < R; c += 16) {
                        float g[16], u[16];
                        tmem_ld16(tg + c, g);
                        tmem_ld16(tg + NT + c, u);
                        if (r < rows) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int tok = c + i;
                                const float h = g[i] / (1.f + expf(-g[i])) * u[i];
                                // K-major, 128-byte swizzle: 16-byte chunk (cin / 8) ^ (tok % 8) of row tok
                                const uint32_t off = tok * 128 + ((((cin >> 3) ^ (tok & 7)) & 7) << 4) + (cin & 7) * 2;
                                *reinterpret_cast<__nv_bfloat16*>(hb + off) = __float2bfloat16_rn(h);
                            }
                        }
                    }
                    fence_proxy_async();  // h is read by the tensor cores (async proxy)
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&aempty[ab]);
                        mbar_arrive(&hready[t]);
                    }
                }
                if (!ok) break;
                // phase B epilogues: Y columns of d -> partial rows
                for (int dc = 0; !UP && dc < nkB; ++dc, ++ny) {
                    const int yb = ny & 1;
                    if (!wait_warp(&yfull[yb], (ny >> 1) & 1, 20)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t ty = tmem_base + lane_off + 4 * NT + yb * NT;
                    float* col = prow + dc * 128 + r;
#pragma unroll 1
                    for (int c = 0; c < NT && c < R; c += 16) {
                        float y[16];
                        tmem_ld16(ty + c, y);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int tok = c + i;
                            if (tok < R) {
                                float* dst = col + (size_t)tok * d;
                                *dst = chunk == 0 ? y[i] : *dst + y[i];
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&yempty[yb]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(C::kTmemCols));
    }
}

template <int NT, bool UP>
static cudaError_t launch_tcd_nt(const TcdLaunch& a, cudaStream_t st) {
    using C = TcdCfg<NT>;
    TcdParams p;
    std::memset(&p, 0, sizeof(p));
    if (encode_bf16_2d(&p.map_x, a.x, a.d, a.T, (uint64_t)a.d * 2, 64, NT) != MOE_OK ||
        encode_bf16_2d(&p.map_x1, a.x, a.d, a.T, (uint64_t)a.d * 2, 64, 1) != MOE_OK)
        return cudaErrorInvalidValue;
    if (NT == 32) {
        cudaError_t e = launch_gather_rows(a.x, a.perm, a.expert_offsets, a.N, a.k, a.d, a.rows_cap, a.x_perm, st);
        if (e != cudaSuccess) return e;
        if (encode_bf16_2d(&p.map_xp, a.x_perm, a.d, a.rows_cap > 0 ? a.rows_cap : 1, (uint64_t)a.d * 2, 64, NT) !=
            MOE_OK)
            return cudaErrorInvalidValue;
    }
    p.perm = a.perm; p.topk = a.k;
    p.table = a.table; p.hdr = a.hdr; p.segs = a.segs; p.partial = a.partial;
    p.u_out = a.u_out; p.d = a.d; p.N = a.N; p.I = a.I; p.err = a.err;
    p.n_prefetch = a.u_out ? 0 : a.prefetch_shared;
    auto kernel = ffn_tcd_kernel<NT, UP>;
    cudaError_t e = allow_max_smem(kernel);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kernel, dim3(a.grid), dim3(kTcdThreads), C::kSmem, st, p);
    return note_launch(reinterpret_cast<const void*>(kernel), kTcdThreads, C::kSmem, e);
}

cudaError_t launch_tcd_ffn(const TcdLaunch& a, cudaStream_t st) {
    if (a.d % 128 != 0) return cudaErrorInvalidValue;
    const bool up = a.u_out != nullptr;
    switch (a.nt) {
        case 16: return up ? launch_tcd_nt<16, true>(a, st) : launch_tcd_nt<16, false>(a, st);
        case 32: return up ? launch_tcd_nt<32, true>(a, st) : launch_tcd_nt<32, false>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe
