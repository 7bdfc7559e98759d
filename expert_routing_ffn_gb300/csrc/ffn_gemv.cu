// Stage 3b, decode-size segments: SwiGLU expert FFN as an HBM-streaming GEMV.
//
// y = sum_i SiLU(x . Wg[i]) (x . Wu[i]) Wd[i, :]  (FloE method §1 with the
// identity mask; weights channel-major [I, d] so that channel i's gate, up
// and down rows are each one contiguous d-vector).
//
// Work split: the channels of every segment (an expert with up to RG token
// rows) form one list, cut into G equal ranges, one per CTA (G = SMs x CTAs
// per SM).  A CTA streams its range in stages of CH channels: one bulk copy
// (TMA engine) per matrix per stage brings the CH gate, up and down rows into
// shared memory, NS stages in flight, completion tracked by mbarriers.  Every
// weight byte is read from HBM exactly once; the token rows are held in
// registers.
//
// Per stage: each thread owns one 16-byte chunk of d; it forms the partial
// gate/up dot products of its chunk for every (channel, row), each warp sums
// them with a reduce-scatter, one block barrier publishes the per-warp sums,
// every warp then forms h = SiLU(g) * u itself and adds h * Wd[channel,
// chunk] into its register accumulators for the output columns of the same
// chunk.  The barrier also proves the previous stage's buffer is free, so
// thread 0 refills it right there (no second barrier per stage).  When a CTA leaves a segment it writes
// its partial output rows; a second kernel sums the partials of each row in a
// fixed order (deterministic, no atomics).
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kNSMax = 8;

// Issues the bulk copies of one CTA's stages, in the order they are read.
// Run by thread 0 only.
struct Producer {
    const Seg* segs;
    const ExpertEntry* table;
    const int32_t* list;  // FloE channel lists
    unsigned char* stage_mem;
    uint64_t* full;
    size_t row_bytes, mat_bytes, stage_bytes;
    int NS, CH, seg, ch, hi, n_seg;
    int issued;
    uint64_t policy;
    // the segment being issued and its expert's weights, loaded once per
    // segment (a dependent global load per stage would sit on the pipeline's
    // critical path)
    int cached;
    int c_start, c_I, c_list_off;
    const char* w[3];

    __device__ __forceinline__ bool done() const { return ch >= hi || seg >= n_seg; }

    __device__ __forceinline__ void load_seg() {
        const Seg S = segs[seg];
        const ExpertEntry& E = table[S.expert];
        c_start = S.ch_start; c_I = S.I; c_list_off = S.list_off;
#pragma unroll
        for (int m = 0; m < 3; ++m) w[m] = static_cast<const char*>(E.w[m]);
        cached = seg;
    }

    __device__ __forceinline__ void issue() {
        if (cached != seg) load_seg();
        const int local = ch - c_start;
        const int seg_end = min(hi, c_start + c_I) - c_start;
        // an up-only stage holds 3 x CH up rows (the whole stage buffer)
        const int nch = min(c_list_off == kUpOnly ? 3 * CH : CH, seg_end - local);
        const int b = issued % NS;
        unsigned char* buf = stage_mem + (size_t)b * stage_bytes;
        const uint32_t bytes = (uint32_t)(nch * row_bytes);
        if (c_list_off == kUpOnly) {
            // FloE first pass: up rows only, 3 x CH of them per stage
            mbar_arrive_expect_tx(&full[b], bytes);
            bulk_g2s(buf, w[1] + (size_t)local * row_bytes, bytes, &full[b], policy);
        } else if (c_list_off >= 0) {
            // FloE: gate and down rows of the listed channels only
            mbar_arrive_expect_tx(&full[b], 2 * bytes);
            // the list entries of the stage are loaded together (nch <= 4)
            int rows[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) rows[c] = c < nch ? list[c_list_off + local + c] : 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (c >= nch) break;
                const size_t row = (size_t)rows[c];
                bulk_g2s(buf + c * row_bytes, w[0] + row * row_bytes, (uint32_t)row_bytes, &full[b], policy);
                bulk_g2s(buf + 2 * mat_bytes + c * row_bytes, w[2] + row * row_bytes, (uint32_t)row_bytes,
                         &full[b], policy);
            }
        } else {
            mbar_arrive_expect_tx(&full[b], 3 * bytes);
#pragma unroll
            for (int m = 0; m < 3; ++m)
                bulk_g2s(buf + m * mat_bytes, w[m] + (size_t)local * row_bytes, bytes, &full[b], policy);
        }
        ch += nch;
        if (ch >= c_start + c_I) ++seg;
        ++issued;
    }
};

template <int V>
__device__ __forceinline__ float dot_v(const float* a, const float* b) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int j = 0; j < V; j += 2) fma2(s0, s1, a[j], a[j + 1], b[j], b[j + 1]);
    return s0 + s1;
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + expf(-g)); }

// Barrier among the block's threads (named barrier 1, separate from the
// __syncthreads used between segment pieces).
__device__ __forceinline__ void consumer_sync(int n_threads) {
    asm volatile("bar.sync 1, %0;" ::"r"(n_threads) : "memory");
}

struct GemvShared {
    uint64_t* full;
    float* red;        // [2][n_warps][32]
    int* abort_flag;
    unsigned char* stage_mem;
    Producer* prod;    // thread 0's copy issuer
};

// One segment piece: channels [llo, lhi) of segment S, ROWS token rows.
template <typename W, int CH, int ROWS, bool FLOE>
__device__ __forceinline__ void gemv_piece(const GemvParams& p, const Seg& S, int llo, int lhi,
                                           int cta, const GemvShared& sh, int n_cons,
                                           int& stage_k) {
    constexpr int V = Vec<W>::n;
    constexpr int NV = 2 * CH * ROWS;
    static_assert(NV <= 32, "per-stage outputs must fit one warp reduce-scatter");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = n_cons >> 5;
    const int d = p.d;
    const size_t row_bytes = (size_t)d * sizeof(W);
    const size_t mat_bytes = (size_t)CH * row_bytes;
    const W* x = static_cast<const W*>(p.x);
    const bool sparse = FLOE && S.list_off >= 0;  // FloE segment: gate/down of listed channels
    const size_t stage_bytes = 3 * mat_bytes;

    float xr[ROWS][V];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const int token = S.expert < p.N ? p.perm[S.row0 + r] / p.topk : S.row0 + r;
        const uint4 raw = reinterpret_cast<const uint4*>(x + (size_t)token * d)[tid];
        unpack16(raw, xr[r], (W*)nullptr);
    }
    float yacc[ROWS][V];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int j = 0; j < V; ++j) yacc[r][j] = 0.f;

    for (int i = llo; i < lhi; i += CH) {
        const int nch = min(CH, lhi - i);
        const int b = stage_k % p.NS;
        const uint32_t par = (uint32_t)((stage_k / p.NS) & 1);
        if (!mbar_wait(&sh.full[b], par)) {
            set_error(p.err, MOE_ERR_TIMEOUT, cta);
            *sh.abort_flag = 1;
        }
        const unsigned char* buf = sh.stage_mem + (size_t)b * stage_bytes;
        // partial gate/up dot products of this thread's 16-byte chunk
        constexpr int NB = NV <= 2 ? 2 : NV <= 4 ? 4 : NV <= 8 ? 8 : NV <= 16 ? 16 : 32;
        constexpr int SH = NB == 2 ? 4 : NB == 4 ? 3 : NB == 8 ? 2 : NB == 16 ? 1 : 0;  // 5 - log2(NB)
        float v[NB];
#pragma unroll
        for (int q = 0; q < NB; ++q) v[q] = 0.f;
#pragma unroll
        for (int cc = 0; cc < CH; ++cc) {
            if (cc < nch) {
                float wg[V];
                unpack16(reinterpret_cast<const uint4*>(buf + cc * row_bytes)[tid], wg, (W*)nullptr);
#pragma unroll
                for (int r = 0; r < ROWS; ++r) v[cc * 2 * ROWS + r] = dot_v<V>(wg, xr[r]);
                if (!sparse) {
                    float wu[V];
                    unpack16(reinterpret_cast<const uint4*>(buf + mat_bytes + cc * row_bytes)[tid], wu,
                             (W*)nullptr);
#pragma unroll
                    for (int r = 0; r < ROWS; ++r) v[cc * 2 * ROWS + ROWS + r] = dot_v<V>(wu, xr[r]);
                }
            }
        }
        // block sum: warp reduce-scatter, one consumer barrier, then every
        // warp reads the per-warp sums (double-buffered by stage parity)
        float* red = sh.red + (size_t)(stage_k & 1) * nw * 32;
        const float t = warp_reduce_scatter<NB>(v);
        if ((lane & ((1 << SH) - 1)) == 0) red[warp * 32 + (lane >> SH)] = t;
        consumer_sync(n_cons);
        // every thread has finished the previous stage, so its buffer can be
        // refilled with the stage NS - 1 ahead of this one
        if (tid == 0 && stage_k > 0 && !sh.prod->done()) sh.prod->issue();
        float hq = 0.f;
        if (lane < CH * ROWS) {
            const int cc = lane / ROWS, r = lane % ROWS;
            float g = 0.f, u = 0.f;
            for (int w = 0; w < nw; ++w) {
                g += red[w * 32 + cc * 2 * ROWS + r];
                u += red[w * 32 + cc * 2 * ROWS + ROWS + r];
            }
            if (FLOE && cc < nch && sparse) {
                // FloE: u from the dense up projection, h only on this row's kept channels
                const int ch = p.floe_list[S.list_off + i + cc];
                const size_t row = (size_t)(S.row0 + r);
                u = p.floe_u[row * p.I + ch];
                const bool keep = (p.floe_kept[row * p.words + (ch >> 5)] >> (ch & 31)) & 1u;
                hq = keep ? silu(g) * u : 0.f;
            } else {
                hq = cc < nch ? silu(g) * u : 0.f;
            }
        }
        // down projection: y[r, chunk] += h[c, r] * Wd[c, chunk]
#pragma unroll
        for (int cc = 0; cc < CH; ++cc) {
            if (cc < nch) {
                float wd[V];
                unpack16(reinterpret_cast<const uint4*>(buf + 2 * mat_bytes + cc * row_bytes)[tid], wd,
                         (W*)nullptr);
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const float h = __shfl_sync(0xffffffffu, hq, cc * ROWS + r);
#pragma unroll
                    for (int j = 0; j < V; j += 2) fma2(yacc[r][j], yacc[r][j + 1], h, h, wd[j], wd[j + 1]);
                }
            }
        }
        ++stage_k;
        if (*sh.abort_flag) break;
    }
    // partial output rows of this CTA for this segment
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        float* dst = p.partial + ((size_t)(S.pbase + (cta - S.c0) * ROWS + r)) * d + (size_t)tid * V;
#pragma unroll
        for (int j = 0; j < V; j += 4)
            *reinterpret_cast<float4*>(dst + j) = make_float4(yacc[r][j], yacc[r][j + 1], yacc[r][j + 2], yacc[r][j + 3]);
    }
}

// FloE first pass over one segment piece: u[row, ch] = x_row . W_up[ch, :]
// for ROWS <= 2 token rows, 3 x CH up rows per stage, no down projection.
template <typename W, int CHU, int ROWS>
__device__ __forceinline__ void gemv_piece_up(const GemvParams& p, const Seg& S, int llo, int lhi,
                                              int cta, const GemvShared& sh, int n_cons, int& stage_k) {
    constexpr int V = Vec<W>::n;
    constexpr int NV = CHU * ROWS;
    static_assert(NV <= 16, "per-stage outputs must fit one 16-value reduce-scatter");
    constexpr int NB = NV <= 2 ? 2 : NV <= 4 ? 4 : NV <= 8 ? 8 : 16;
    constexpr int SH = NB == 2 ? 4 : NB == 4 ? 3 : NB == 8 ? 2 : 1;  // 5 - log2(NB)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = n_cons >> 5;
    const int d = p.d;
    const size_t row_bytes = (size_t)d * sizeof(W);
    const size_t stage_bytes = (size_t)CHU * row_bytes;
    const W* x = static_cast<const W*>(p.x);
    float xr[ROWS][V];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const int token = p.perm[S.row0 + r] / p.topk;
        unpack16(reinterpret_cast<const uint4*>(x + (size_t)token * d)[tid], xr[r], (W*)nullptr);
    }
    for (int i = llo; i < lhi; i += CHU) {
        const int nch = min(CHU, lhi - i);
        const int b = stage_k % p.NS;
        if (!mbar_wait(&sh.full[b], (uint32_t)((stage_k / p.NS) & 1))) {
            set_error(p.err, MOE_ERR_TIMEOUT, cta);
            *sh.abort_flag = 1;
        }
        const unsigned char* buf = sh.stage_mem + (size_t)b * stage_bytes;
        float v[NB];
#pragma unroll
        for (int q = 0; q < NB; ++q) v[q] = 0.f;
#pragma unroll
        for (int cc = 0; cc < CHU; ++cc) {
            if (cc < nch) {
                float wu[V];
                unpack16(reinterpret_cast<const uint4*>(buf + cc * row_bytes)[tid], wu, (W*)nullptr);
#pragma unroll
                for (int r = 0; r < ROWS; ++r) v[cc * ROWS + r] = dot_v<V>(wu, xr[r]);
            }
        }
        float* red = sh.red + (size_t)(stage_k & 1) * nw * 32;
        const float t = warp_reduce_scatter<NB>(v);
        if ((lane & ((1 << SH) - 1)) == 0) red[warp * 32 + (lane >> SH)] = t;
        consumer_sync(n_cons);
        if (tid == 0 && stage_k > 0 && !sh.prod->done()) sh.prod->issue();
        if (warp == 0 && lane < CHU * ROWS) {
            const int cc = lane / ROWS, r = lane % ROWS;
            if (cc < nch) {
                float u = 0.f;
                for (int w = 0; w < nw; ++w) u += red[w * 32 + lane];
                p.floe_u[(size_t)(S.row0 + r) * p.I + i + cc] = u;
            }
        }
        ++stage_k;
        if (*sh.abort_flag) break;
    }
}

// Block = one thread per 16-byte chunk of d.  Thread 0 also issues the
// stage copies.
template <typename W, int RG, int CH, int MAXT, bool FLOE>
__device__ __forceinline__ void ffn_gemv_body(const GemvParams& p) {
    __shared__ __align__(8) uint64_t full[kNSMax];
    __shared__ float red_s[2 * (MAXT / 32) * 32];
    __shared__ int s_abort;
    extern __shared__ __align__(128) unsigned char stage_mem[];

    const int tid = threadIdx.x;
    const int n_cons = blockDim.x;
    if (!FLOE && tid < 32 && p.prefetch_shared > 0)
        l2_prefetch_shared_experts(p.table, p.N, p.prefetch_shared, p.d, (int)sizeof(W), blockIdx.x, gridDim.x, tid);
    grid_dep_wait();  // the plan and perm come from the previous kernels
    const PlanHeader hdr = *p.hdr;
    const int cta = blockIdx.x;
    if (cta >= hdr.G) return;
    const int lo = cta * hdr.P, hi = min(lo + hdr.P, hdr.total_ch);
    if (lo >= hi || hdr.n_seg <= 0) return;
    const size_t row_bytes = (size_t)p.d * sizeof(W);

    int s_lo = 0, s_hi = hdr.n_seg - 1;
    while (s_lo < s_hi) {
        const int mid = (s_lo + s_hi + 1) >> 1;
        if (p.segs[mid].ch_start <= lo) s_lo = mid; else s_hi = mid - 1;
    }
    const int seg0 = s_lo;

    const int NSx = p.NS;
    Producer prod;
    if (tid == 0) {
        for (int b = 0; b < NSx; ++b) mbar_init(&full[b], 1);
        fence_mbar_init();
        s_abort = 0;
        prod.segs = p.segs; prod.table = p.table; prod.list = p.floe_list; prod.stage_mem = stage_mem;
        prod.full = full;
        prod.row_bytes = row_bytes; prod.mat_bytes = CH * row_bytes;
        prod.stage_bytes = 3 * CH * row_bytes; prod.NS = NSx; prod.CH = CH;
        prod.seg = seg0;
        prod.ch = lo; prod.hi = hi; prod.n_seg = hdr.n_seg; prod.issued = 0; prod.cached = -1;
        prod.policy = l2_evict_first_policy();
        // fill every buffer but the one the first refill will use
        for (int k = 0; k < NSx && !prod.done(); ++k) prod.issue();
    }
    __syncthreads();

    GemvShared sh;
    sh.full = full; sh.red = red_s; sh.abort_flag = &s_abort; sh.stage_mem = stage_mem; sh.prod = &prod;
    int stage_k = 0;
    int seg = seg0, ch = lo;
    while (ch < hi && seg < hdr.n_seg) {
        const Seg S = p.segs[seg];
        const int llo = ch - S.ch_start;
        const int lhi = min(hi, S.ch_start + S.I) - S.ch_start;
        if (FLOE && S.list_off == kUpOnly) {
            // (the up-only pass runs on the CH = 2 instantiation; the sparse
            // pass's wider stages carry no up-only segments)
            if constexpr (3 * CH * 2 <= 16) {
                if (S.rows == 1) gemv_piece_up<W, 3 * CH, 1>(p, S, llo, lhi, cta, sh, n_cons, stage_k);
                else if (S.rows == 2) gemv_piece_up<W, 3 * CH, 2>(p, S, llo, lhi, cta, sh, n_cons, stage_k);
                else { if (tid == 0) set_error(p.err, MOE_ERR_DEVICE_INDEX, seg); s_abort = 1; }
            } else {
                if (tid == 0) set_error(p.err, MOE_ERR_DEVICE_INDEX, seg);
                s_abort = 1;
            }
        } else switch (S.rows) {
#define MOE_PIECE(R)                                                                        \
    case R:                                                                                 \
        if (R <= RG) {                                                                      \
            gemv_piece<W, CH, (R <= RG ? R : 1), FLOE>(p, S, llo, lhi, cta, sh, n_cons, stage_k); \
        } else {                                                                            \
            if (tid == 0) set_error(p.err, MOE_ERR_DEVICE_INDEX, seg);                      \
            s_abort = 1;                                                                    \
        }                                                                                   \
        break;
            MOE_PIECE(1) MOE_PIECE(2) MOE_PIECE(3) MOE_PIECE(4)
            MOE_PIECE(5) MOE_PIECE(6) MOE_PIECE(7) MOE_PIECE(8)
#undef MOE_PIECE
            default:
                if (tid == 0) set_error(p.err, MOE_ERR_DEVICE_INDEX, seg);
                s_abort = 1;
        }
        __syncthreads();
        if (*(volatile int*)&s_abort) break;
        ch = S.ch_start + lhi;
        ++seg;
    }
    // after an abort, wait (bounded) for the copies still in flight before
    // the CTA exits and its shared memory is released
    if (tid == 0 && s_abort) {
        for (int k = stage_k; k < prod.issued; ++k)
            (void)mbar_wait(&full[k % NSx], (uint32_t)((k / NSx) & 1));
    }
}

// The register file is split over the SM's four sub-partitions, each taking
// a quarter of the resident warps: 16 warps per SM allow 128 registers per
// thread.  Two CTAs of 256 threads per SM (d <= 2048) ...
template <typename W, int RG, int CH, bool FLOE>
__global__ void __launch_bounds__(256, 2) ffn_gemv_kernel_x2(GemvParams p) {
    ffn_gemv_body<W, RG, CH, 256, FLOE>(p);
}

// ... or one CTA of up to 512 threads (d <= 4096).
template <typename W, int RG, int CH, bool FLOE>
__global__ void __launch_bounds__(512, 1) ffn_gemv_kernel_x1(GemvParams p) {
    ffn_gemv_body<W, RG, CH, 512, FLOE>(p);
}

// Sum the partial rows of each output row (in the order of partial_item_runs
// and unit_table_sum).  The row's segment rows ("units": one for a y_perm
// row, one per shared expert for a y_shared row) are looked up by warp 0.
// direct = 0 (GEMV partials, up to a few hundred pieces a segment): block =
// one output row x 32 float4 columns of d; all warps sum the units' runs into
// dynamic shared memory (max(1, n_shared) * kSumChunks * 32 float4), then warp
// 0 adds them up.  direct = 1 (decode tensor-core partials, a few pieces a
// segment): block = one output row x 256 float4 columns, one thread per
// column sums its units alone (partial_unit_sum, the same arithmetic).
__global__ void __launch_bounds__(256) gemv_reduce_kernel(const PlanHeader* __restrict__ hdr_p,
                                                          const Seg* __restrict__ segs,
                                                          const int32_t* __restrict__ seg_first,
                                                          const int32_t* __restrict__ expert_offsets,
                                                          const float* __restrict__ partial, int d,
                                                          int N, int n_shared, int T, int routed_cap,
                                                          float* __restrict__ y_perm,
                                                          float* __restrict__ y_shared, int direct) {
    __shared__ UnitTable U;
    extern __shared__ float4 s_runs[];
    grid_dep_wait();
    const int row = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool routed = row < routed_cap;
    if (!routed && (row - routed_cap >= T || n_shared == 0)) return;
    if (warp == 0) {
        // lane 0: the routed row's segment; lane s < n_shared: shared expert s
        const PlanHeader& hdr = *hdr_p;
        bool has = false;
        Seg S;
        int srow = 0;
        if (routed) {
            if (row < hdr.n_routed_rows) {
                // expert e with offsets[e] <= row < offsets[e+1]: offsets are
                // non-decreasing from 0, so e = #{e < N : offsets[e] <= row} - 1
                const bool lo = lane < N && expert_offsets[lane] <= row;
                const bool hi = lane + 32 < N && expert_offsets[lane + 32] <= row;
                const int e = __popc(__ballot_sync(0xffffffffu, lo)) + __popc(__ballot_sync(0xffffffffu, hi)) - 1;
                if (lane == 0 && e >= 0) {
                    const int local = row - expert_offsets[e];
                    const int si = seg_first[e] + local / hdr.rg;
                    if (si >= 0 && si < hdr.n_seg) {
                        S = segs[si]; srow = local % hdr.rg;
                        has = seg_row_ok(S, srow, hdr.n_partial_rows);
                    }
                }
            }
        } else if (lane < n_shared) {
            const int t = row - routed_cap;
            const int si = seg_first[N + lane] + t / hdr.rg;
            if (si >= 0 && si < hdr.n_seg) {
                S = segs[si]; srow = t % hdr.rg;
                has = seg_row_ok(S, srow, hdr.n_partial_rows);
            }
        }
        unit_table_publish(U, has, S, srow);
    }
    __syncthreads();
    // a routed row past the computed rows, or a bad plan entry (error word set
    // by the plan): nothing to write
    if (routed && U.n == 0) return;
    float* out = routed ? y_perm + (size_t)row * d : y_shared + (size_t)(row - routed_cap) * d;
    if (direct) {
        const int q = blockIdx.y * blockDim.x + threadIdx.x;
        if (q >= d / 4) return;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int u = 0; u < U.n; ++u) {
            const float4 y = partial_unit_sum(partial, U.seg[u], U.row[u], d, q);
            if (routed) acc = y; else add4(acc, y);
        }
        reinterpret_cast<float4*>(out)[q] = acc;
        return;
    }
    const int q = blockIdx.y * 32 + lane;
    const bool col_ok = q < d / 4;
    if (col_ok) unit_table_runs(U, partial, d, q, s_runs, warp, blockDim.x >> 5);
    __syncthreads();
    if (warp != 0 || !col_ok) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int u = 0; u < U.n; ++u) {
        const float4 y = unit_table_sum(U, u, s_runs);
        if (routed) acc = y; else add4(acc, y);
    }
    reinterpret_cast<float4*>(out)[q] = acc;
}

// ---------------------------------------------------------------------------
// Instantiations: bf16 with d <= 2048 runs 2 CTAs per SM, larger d one CTA
// per SM; 4 rows per segment for bf16 (gemv_rows), 8 for the small fp32 layer.
template <typename K>
static cudaError_t launch_gemv_k(K kernel, int maxt, int vec, int ch, int esize, const GemvParams& p,
                                 int G, cudaStream_t st) {
    const int threads = p.d / vec;
    if (threads > maxt || threads % 32) return cudaErrorInvalidValue;
    const size_t smem = (size_t)p.NS * 3 * ch * p.d * esize;
    cudaError_t e = allow_max_smem(kernel);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kernel, dim3(G), dim3(threads), smem, st, p);
    return note_launch(reinterpret_cast<const void*>(kernel), threads, smem, e);
}

static int gemv_ctas_per_sm(int d, bool bf16) {
#ifdef MOE_XP_GEMV_ONE_CTA
    if (bf16) return 1;
#endif
    return (bf16 && d <= 2048) || !bf16 ? 2 : 1;
}

int gemv_grid_for(int d, bool bf16, int sms) {
    const int g = sms * gemv_ctas_per_sm(d, bf16);
    return g > kGemvMaxCtas ? kGemvMaxCtas : g;
}

int gemv_stages(int d, bool bf16, int ch) {
    const size_t stage = (size_t)3 * ch * d * (bf16 ? 2 : 4);
    const size_t budget = gemv_ctas_per_sm(d, bf16) == 2 ? 100 * 1024 : 200 * 1024;
    int ns = (int)(budget / stage);
    return ns < 2 ? 2 : (ns > kNSMax ? kNSMax : ns);
}

// floe = true selects the instantiation with the FloE modes (up-only and
// sparse segments); the dense instantiation carries none of their code.
// sparse = true: FloE's second pass (gate / down of the listed channels), 4
// channels per stage, so a block barrier serves twice the bytes (p.NS from
// gemv_stages(d, bf16, 4)).
cudaError_t launch_gemv(const GemvParams& p, int G, bool bf16, cudaStream_t st, bool floe, bool sparse) {
    if (bf16 && floe && sparse) {
        if (p.d <= 2048) return launch_gemv_k(ffn_gemv_kernel_x2<__nv_bfloat16, 4, 4, true>, 256, 8, 4, 2, p, G, st);
        return launch_gemv_k(ffn_gemv_kernel_x1<__nv_bfloat16, 4, 4, true>, 512, 8, 4, 2, p, G, st);
    }
    if (bf16) {
#ifdef MOE_XP_GEMV_ONE_CTA
        if (false)
#else
        if (p.d <= 2048)
#endif
            return floe ? launch_gemv_k(ffn_gemv_kernel_x2<__nv_bfloat16, 4, 2, true>, 256, 8, 2, 2, p, G, st)
                        : launch_gemv_k(ffn_gemv_kernel_x2<__nv_bfloat16, 4, 2, false>, 256, 8, 2, 2, p, G, st);
        return floe ? launch_gemv_k(ffn_gemv_kernel_x1<__nv_bfloat16, 4, 2, true>, 512, 8, 2, 2, p, G, st)
                    : launch_gemv_k(ffn_gemv_kernel_x1<__nv_bfloat16, 4, 2, false>, 512, 8, 2, 2, p, G, st);
    }
    return launch_gemv_k(ffn_gemv_kernel_x2<float, 8, 2, false>, 256, 4, 2, 4, p, G, st);
}

cudaError_t launch_gemv_reduce(const GemvReduceArgs& a, cudaStream_t st) {
    const int rows = a.routed_cap + (a.n_shared > 0 ? a.T : 0);
    if (rows == 0) return cudaSuccess;
    const int cols = a.direct ? 256 : 32;  // float4 columns per block
    dim3 grid(rows, (a.d / 4 + cols - 1) / cols);
    const size_t smem =
        a.direct ? 0 : (size_t)(a.n_shared > 1 ? a.n_shared : 1) * kSumChunks * 32 * sizeof(float4);
    return launch_pdl(gemv_reduce_kernel, grid, dim3(256), smem, st, a.hdr, a.segs, a.seg_first, a.expert_offsets,
                      a.partial, a.d, a.N, a.n_shared, a.T, a.routed_cap, a.y_perm, a.y_shared, a.direct ? 1 : 0);
}

}  // namespace moe
