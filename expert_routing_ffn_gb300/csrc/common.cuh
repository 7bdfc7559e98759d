// Shared device helpers for the sm_103a MoE layer kernels: PTX wrappers for
// mbarriers and bulk (TMA) copies, the device error word, bf16 unpacking,
// and the workspace / FFN-plan layout used by the host launchers and the
// kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------- constants
constexpr int kMaxExperts = 64;       // expert sets are uint64 bitmasks
constexpr int kMaxTopK = 8;
constexpr int kMaxShared = 8;         // shared experts per layer
constexpr int kGemvMaxRows = 8;       // rows per GEMV segment (register-resident)
constexpr int kGemvMaxCtas = 512;     // upper bound of the GEMV grid (workspace sizing)
constexpr int kAlign = 256;
constexpr int kPermChunk = 1024;      // slots per block of the multi-block permutation
// Iteration bound of every spin wait; a wait that exceeds it records
// MOE_ERR_TIMEOUT and gives up instead of hanging the GPU.
constexpr uint32_t kSpinLimit = 1u << 24;

// ---------------------------------------------------------------- error word
struct DevError {
    int code;
    int detail;
    int pad[14];
};

__device__ __forceinline__ void set_error(DevError* e, int code, int detail) {
    if (atomicCAS(&e->code, 0, code) == 0) e->detail = detail;
}

// ---------------------------------------------------------------- FFN plan
// One GEMV segment: up to kGemvMaxRows rows that share one expert's weights.
// Its I channels occupy [ch_start, ch_start + I) of the global channel list,
// which is split evenly over the G CTAs of the GEMV grid (P channels each).
// CTA c writes a partial [rows, d] sum for every segment it overlaps at
// partial row pbase + (c - c0) * rows.
struct alignas(16) Seg {
    int expert;     // 0..N-1 routed, N + s shared expert s
    int row0;       // routed: first permuted position; shared: first token
    int rows;
    int I;
    int ch_start;
    int c0;         // first CTA that covers this segment
    int npieces;
    int pbase;      // first partial row
    int list_off;   // FloE: offset of this expert's channel list (-1: dense, channels 0..I-1;
                    // kUpOnly: dense up projection only, u written to the workspace)
};
constexpr int kUpOnly = -2;

struct PlanHeader {
    int n_seg;
    int total_ch;
    int P;          // channels per CTA
    int G;          // GEMV grid
    int rg;         // rows per segment
    int n_partial_rows;
    int n_routed_rows;
    int pad[9];
};

// The partial rows of one (segment, row) are summed in one fixed two-level
// order, shared by every kernel that reduces them so that their results agree
// bitwise: the segment's pieces form at most kSumChunks runs of
// ceil(npieces / kSumChunks) consecutive pieces; each run is summed in piece
// order from zero, then the run sums are added in run order from zero.  The
// runs are independent, so different warps sum them at once: a row spread over
// a few hundred CTAs then costs a few dependent L2 round trips, not one per
// piece.  A work item is a group of consecutive runs of at most eight pieces
// in all (or one longer run), whose loads are all in flight together.
constexpr int kSumChunks = 8;
__device__ __forceinline__ int sum_run_len(int npieces) { return (npieces + kSumChunks - 1) / kSumChunks; }
__device__ __forceinline__ int sum_runs(int npieces) {
    const int c = sum_run_len(npieces);
    return c > 0 ? (npieces + c - 1) / c : 0;
}
__device__ __forceinline__ int sum_runs_per_item(int npieces) {
    const int c = sum_run_len(npieces);
    return c >= 8 ? 1 : 8 / c;
}
__device__ __forceinline__ int sum_items(int npieces) {
    const int rpi = sum_runs_per_item(npieces);
    return (sum_runs(npieces) + rpi - 1) / rpi;
}
__device__ __forceinline__ void add4(float4& a, const float4& b) {
    a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
}
// Item `item` of segment S, row `row`, float4 column q of d: each of its runs'
// sums goes to runs[c * 32] (c = run index).
__device__ __forceinline__ void partial_item_runs(const float* __restrict__ partial, const Seg& S, int row,
                                                  int d, int q, int item, float4* runs) {
    const int len = sum_run_len(S.npieces), rpi = sum_runs_per_item(S.npieces);
    int run = item * rpi;
    const int p_end = min((run + rpi) * len, S.npieces);
    const float4* base = reinterpret_cast<const float4*>(partial + (size_t)(S.pbase + row) * d) + q;
    const size_t step = (size_t)S.rows * (size_t)(d / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int left = len;  // pieces still to add to the current run
    for (int p = run * len; p < p_end; p += 8) {
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (p + i < p_end) v[i] = __ldcg(base + (size_t)(p + i) * step);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (p + i < p_end) {
                add4(acc, v[i]);
                if (--left == 0 || p + i + 1 == p_end) {
                    runs[run * 32] = acc;
                    acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    left = len;
                    ++run;
                }
            }
        }
    }
}
// The same sum of one whole (segment, row) by one thread: its runs' sums are
// added as they complete, which is unit_table_sum's arithmetic.  For segments
// of few pieces (the decode tensor-core path), where one thread per column
// has all the loads in flight anyway.
__device__ __forceinline__ float4 partial_unit_sum(const float* __restrict__ partial, const Seg& S, int row,
                                                   int d, int q) {
    const int len = sum_run_len(S.npieces), np = S.npieces;
    const float4* base = reinterpret_cast<const float4*>(partial + (size_t)(S.pbase + row) * d) + q;
    const size_t step = (size_t)S.rows * (size_t)(d / 4);
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f), acc = y;
    int left = len;
    for (int p = 0; p < np; p += 8) {
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (p + i < np) v[i] = __ldcg(base + (size_t)(p + i) * step);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (p + i < np) {
                add4(acc, v[i]);
                if (--left == 0 || p + i + 1 == np) {
                    add4(y, acc);
                    acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    left = len;
                }
            }
        }
    }
    return y;
}
// A segment row's partial rows are all inside the partial buffer.
__device__ __forceinline__ bool seg_row_ok(const Seg& S, int row, int n_partial_rows) {
    return S.npieces > 0 && S.pbase + (S.npieces - 1) * S.rows + row < n_partial_rows;
}
// Segment rows ("units") that feed one output, as a block sums them.  Warp 0
// publishes them (lane order = unit order; `has`: this lane holds one) with
// the first work item of each; then every warp takes items round robin.
constexpr int kMaxUnits = kMaxTopK + kMaxShared;
struct UnitTable {
    Seg seg[kMaxUnits];
    int row[kMaxUnits];
    int item0[kMaxUnits + 1];
    int n;
};
__device__ __forceinline__ int unit_table_publish(UnitTable& U, bool has, const Seg& S, int row) {
    const int lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t ub = __ballot_sync(0xffffffffu, has);
    const int u = __popc(ub & lt);
    const int items = has ? sum_items(S.npieces) : 0;
    int incl = items;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (has) { U.seg[u] = S; U.row[u] = row; U.item0[u] = incl - items; }
    if (lane == 31) { U.n = __popc(ub); U.item0[__popc(ub)] = incl; }
    return has ? u : -1;
}
// Sum the runs of every item of the table into runs[(u * kSumChunks + c) * 32 + lane],
// the items taken round robin by warps w = 0..nw-1 (this one: w).
__device__ __forceinline__ void unit_table_runs(const UnitTable& U, const float* __restrict__ partial, int d,
                                                int q, float4* runs, int w, int nw) {
    const int lane = threadIdx.x & 31;
    const int n_items = U.item0[U.n];
    for (int i = w; i < n_items; i += nw) {
        int u = 0;
        while (u + 1 < U.n && U.item0[u + 1] <= i) ++u;
        partial_item_runs(partial, U.seg[u], U.row[u], d, q, i - U.item0[u],
                          runs + (size_t)u * kSumChunks * 32 + lane);
    }
}
// Unit u's sum: its runs in order, from zero.
__device__ __forceinline__ float4 unit_table_sum(const UnitTable& U, int u, const float4* runs) {
    const int lane = threadIdx.x & 31;
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    const int nr = sum_runs(U.seg[u].npieces);
    for (int c = 0; c < nr; ++c) add4(y, runs[((size_t)u * kSumChunks + c) * 32 + lane]);
    return y;
}

// Tensor-core (prefill) plan: one segment per routed expert with rows, plus
// one segment for all shared experts (their channels stacked).  Phase-1
// tiles of a segment: m_tiles x n1 (128-channel tiles), phase-2 tiles:
// m_tiles x d/256; tile index = first tile + nt * m_tiles + mt.
struct TcSeg {
    int shared, expert, row0, rows, m_tiles, n1, tile1, tile2;
    int mbase;  // index of this segment's first (segment, row tile) dependency counter
    // the same tiles at CTA-pair granularity (256-row tiles of a 2-CTA MMA):
    // m_pairs = ceil(rows / 256), first phase-1 / phase-2 pair tile
    int m_pairs, tile1p, tile2p;
};
struct TcPlan {
    int n_seg, n_tiles1, n_tiles2;
    int n_mt;  // (segment, row tile) pairs: the dependency counters in use
    int n_tiles1p, n_tiles2p;  // pair tiles of the two phases
    int pad[10];
    TcSeg seg[kMaxExperts + 1];
};

// Batches above this many tokens run the expert FFN on the tensor cores
// (bf16 layers whose I, I_shared are multiples of 128).
constexpr int kTcMinTokens = 64;

__host__ __device__ inline bool tc_usable(const moe_dims& D) {
    return D.wtype == MOE_DTYPE_BF16 && D.I % 128 == 0 && (D.n_shared == 0 || D.I_shared % 128 == 0) &&
           D.d % 256 == 0;
}
__host__ __device__ inline bool use_tc(const moe_dims& D) { return tc_usable(D) && D.T > kTcMinTokens; }

// Decode-size batches of bf16 layers whose d is a multiple of 128 and whose
// expert widths are multiples of 16 run the dense expert FFN on the tensor
// cores too, with the weight rows as the MMA's M side and the (few) token
// rows of a segment as its N side.
#ifndef MOE_DECODE_TC
#define MOE_DECODE_TC 1
#endif
__host__ __device__ inline bool tcd_shapes(const moe_dims& D) {
    return MOE_DECODE_TC && D.wtype == MOE_DTYPE_BF16 && D.d % 128 == 0 && D.I % 16 == 0 &&
           (D.n_shared == 0 || D.I_shared % 16 == 0);
}
// 1..3 tokens stay on the CUDA-core GEMV, which streams faster at one or two
// rows per expert (the tensor-core path pays a pipeline fill per CTA piece).
constexpr int kTcdMinTokens = 4;
__host__ __device__ inline bool tcd_usable(const moe_dims& D) {
    return tcd_shapes(D) && !use_tc(D) && D.T >= kTcdMinTokens;
}
// Token rows per segment on that path (the MMA's N): up to 32 tokens every
// expert's rows of the batch fit one segment, so each weight is read once.
__host__ __device__ inline int tcd_rows(int T) { return T <= 16 ? 16 : 32; }
constexpr int kTcdMaxCtas = 160;  // grid of that path: min(SMs, kTcdMaxCtas)

// ---------------------------------------------------------------- workspace
struct WsLayout {
    size_t err, ticket, logits_r, logits_p, score, route_part, qp, res_part, plan_hdr, segs, seg_first, perm_counts, lore_z,
        lore_off, lore_list, lore_pos, lore_counts, lore_zp, lore_v, tc_plan, tc_dep,
        x_perm, h_routed, h_shared, floe_u, floe_kept, floe_list, floe_count, partial, total;
    int max_segs, max_partial_rows;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Token rows per GEMV segment (the token rows of a segment stay in registers;
// 4 rows keep a bf16 GEMV thread within the register budget of two CTAs per
// SM).  The workspace sizing and the launch both take it from here.
__host__ __device__ inline int gemv_rows(const moe_dims& D) {
    return D.wtype == MOE_DTYPE_BF16 ? 4 : 8;
}

__host__ __device__ inline WsLayout ws_layout(const moe_dims& D) {
    WsLayout L;
    const size_t T = (size_t)(D.T > 0 ? D.T : 1), N = (size_t)D.N;
    const bool tc = use_tc(D);
    // the GEMV (and its partial sums) only serves batches of <= kTcMinTokens
    // tokens when the tensor-core path takes the larger ones
    const size_t Tg = tc ? (size_t)kTcMinTokens : T;
    const size_t rows_routed = Tg * (size_t)D.k;
    const size_t rows_shared = Tg * (size_t)D.n_shared;
    const int rg = gemv_rows(D);
    // a workspace sized for T serves every batch of at most T tokens: the
    // decode tensor-core path may run for any of them up to kTcMinTokens
    const bool tcd = tcd_shapes(D);
    const int rg_tcd = tcd ? tcd_rows((int)(T < (size_t)kTcMinTokens ? T : (size_t)kTcMinTokens)) : 0;
    // segments: sum over experts of ceil(rows_e / rg) <= rows / rg + N, plus the
    // shared experts' ceil(T / rg) each (the smallest rg gives the most)
    L.max_segs = (int)(rows_routed / rg + N + (size_t)D.n_shared * (T / rg + 1) + 8);
    // the FloE up-only pass plans 2 rows per segment: sum_e ceil(rows_e / 2)
    const int up_segs = (int)(rows_routed / 2 + N + 8);
    if (up_segs > L.max_segs) L.max_segs = up_segs;
    // partial rows: sum over segments of pieces * rows <= rg * G + 2 * all rows
    // (a segment of I channels spans at most I / P + 2 CTA ranges, P >= total / G)
    const size_t spread = (size_t)rg * kGemvMaxCtas > (size_t)rg_tcd * kTcdMaxCtas
                              ? (size_t)rg * kGemvMaxCtas : (size_t)rg_tcd * kTcdMaxCtas;
    L.max_partial_rows = (int)(spread + 2 * (rows_routed + rows_shared) + 16);
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, kAlign); return at; };
    L.err = take(sizeof(DevError));
    L.ticket = take(64);  // arrival counters of last-block-finishes kernels (left at 0)
    L.logits_r = take(T * N * 4);
    L.logits_p = take(T * N * 4);
    L.score = take(T * 4);
    // split-d partial logits of the tensor-core router (bf16 batches of more
    // than kTcMinTokens tokens): up to 8 splits x T x 2N fp32
    L.route_part = take(D.wtype == MOE_DTYPE_BF16 && D.T > kTcMinTokens ? 8 * T * 2 * N * 4 : 0);
    L.qp = take(T * N * 4);
    L.res_part = take(32 * kMaxExperts * 4);  // partial sums of the batch resident set
    L.plan_hdr = take(sizeof(PlanHeader));
    L.segs = take((size_t)L.max_segs * sizeof(Seg));
    L.seg_first = take((N + (size_t)D.n_shared + 1) * 4);
    // per 1024-slot chunk and expert: slot counts of the multi-block permutation
    L.perm_counts = take((T * (size_t)D.k + kPermChunk - 1) / kPermChunk * kMaxExperts * 4);
    L.lore_z = take(T * (size_t)D.k * (size_t)(D.r > 0 ? D.r : 1) * 4);
    // LoRE slots grouped by expert and their B_e z rows (batches of more than
    // kTcMinTokens tokens: the condition of lore_grouped_usable)
    const bool lore_grouped = D.r > 0 && D.T > kTcMinTokens;
    L.lore_off = take(lore_grouped ? (N + 1) * 4 : 0);
    L.lore_list = take(lore_grouped ? T * D.k * 4 : 0);
    L.lore_pos = take(lore_grouped ? T * D.k * 4 : 0);
    L.lore_counts = take(lore_grouped ? (T * (size_t)D.k + kPermChunk - 1) / kPermChunk * kMaxExperts * 4 : 0);
    L.lore_zp = take(lore_grouped ? 8 * T * (size_t)D.k * (size_t)(D.r > 0 ? D.r : 1) * 4 : 0);  // 8 d-splits
    L.lore_v = take(lore_grouped ? T * (size_t)D.k * (size_t)D.d * 4 : 0);
    L.tc_plan = take(sizeof(TcPlan));
    // per (segment, row tile) counters of the prefill FFN's phase dependency
    L.tc_dep = take(tc ? ((T + T * D.k) / 128 + N + 4) * 4 : 0);
    L.x_perm = take(tc || tcd ? T * D.k * (size_t)D.d * 2 : 0);
    L.h_routed = take(tc ? T * D.k * (size_t)D.I * 2 : 0);
    L.h_shared = take(tc ? T * (size_t)D.n_shared * D.I_shared * 2 : 0);
    // FloE (decode batches only)
    L.floe_u = take(rows_routed * (size_t)D.I * 4);
    L.floe_kept = take(rows_routed * (size_t)((D.I + 31) / 32) * 4);
    L.floe_list = take(N * (size_t)D.I * 4);
    L.floe_count = take(N * 4);
    L.partial = take((size_t)L.max_partial_rows * (size_t)D.d * 4);
    L.total = o;
    return L;
}

template <typename Tp>
__host__ __device__ inline Tp* ws_at(void* ws, size_t off) {
    return reinterpret_cast<Tp*>(static_cast<char*>(ws) + off);
}

// ---------------------------------------------------------------- expert table
// Device-resident; filled by moe_expert_table_init.  Entry e < N: routed
// expert e; entry N + s: shared expert s.
struct alignas(64) ExpertEntry {
    const void* w[3];   // gate, up, down: [I, d] each
    int I;
    int pad[9];
    // TMA descriptors (tensor maps) for the tensor-core path: gate/up tiles
    // (K-major) and down tiles (MN-major).
    alignas(64) unsigned char tmap[3][128];
    // The decode tensor-core path: gate, up and down in boxes of 16 rows x 64
    // values (its channel ranges are multiples of 16).
    alignas(64) unsigned char tmap_dec[3][128];
};

// ---------------------------------------------------------------- launch setup
// Raise a kernel's dynamic shared-memory limit to the device maximum, once per
// (kernel, device); later calls (for example inside a stream capture) only
// look the pair up.
cudaError_t allow_max_smem_impl(const void* kernel);

template <typename K>
inline cudaError_t allow_max_smem(K kernel) {
    return allow_max_smem_impl(reinterpret_cast<const void*>(kernel));
}

// ---------------------------------------------------------------- bf16
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

template <typename W> struct Vec;
template <> struct Vec<__nv_bfloat16> { static constexpr int n = 8; };
template <> struct Vec<float> { static constexpr int n = 4; };

// 16 bytes of weights -> fp32 values
__device__ __forceinline__ void unpack16(const uint4& v, float* f, __nv_bfloat16*) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}
__device__ __forceinline__ void unpack16(const uint4& v, float* f, float*) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}

__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(float v) { return v; }

// packed fp32 FMA (two lanes per instruction on sm_100+)
__device__ __forceinline__ void fma2(float& a0, float& a1, float x0, float x1, float y0, float y1) {
    unsigned long long acc, xv, yv;
    asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(xv) : "f"(x0), "f"(x1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(yv) : "f"(y0), "f"(y1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(xv), "l"(yv));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(acc));
}

// ---------------------------------------------------------------- PTX: mbarrier / bulk copy
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Non-blocking probe: true when the phase of the given parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait: returns false after kSpinLimit unsuccessful tries or about
// one second of wall-clock time (%globaltimer, ns), whichever comes first.
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
constexpr uint64_t kWaitNs = 1000000000ull;
#ifndef MOE_WAIT_POLL
#define MOE_WAIT_POLL 0
#endif
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1; i < kSpinLimit; ++i) {
        if (MOE_WAIT_POLL ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 0 && global_ns() - t0 > kWaitNs) return false;
    }
    return false;
}

// 1-D bulk copy global -> shared (TMA engine), completion on an mbarrier.
// src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- dependent launch
// A kernel launched with programmatic stream serialization (launch_pdl) may
// start while the previous kernel on its stream is still running: it calls
// grid_dep_wait() before reading anything that kernel writes (a no-op when
// launched normally).  grid_dep_launch() lets the next such kernel start its
// prologue early.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

// The shared experts' weights do not depend on routing: an FFN kernel that
// starts while the routing kernel still runs (dependent launch) can pull its
// 1/G share of them into L2 before grid_dep_wait(), with HBM otherwise idle.
// One warp issues untracked bulk prefetches of at most 32 KB; every matrix
// holds I * d elements with d a multiple of 64, so each piece is a multiple
// of 16 bytes at a 16-byte aligned address.
__device__ __forceinline__ void l2_prefetch_shared_experts(const ExpertEntry* table, int N, int n_shared, int d,
                                                           int esize, int cta, int G, int lane) {
    constexpr size_t kPiece = 32768;
    for (int s = 0; s < n_shared; ++s) {
        const ExpertEntry& E = table[N + s];
        const size_t bytes = (size_t)E.I * d * esize;
        const size_t share = ((bytes + (size_t)G - 1) / G + 15) & ~(size_t)15;
        const size_t lo = (size_t)cta * share, hi = min(lo + share, bytes);
        for (int m = 0; m < 3; ++m) {
            const char* base = static_cast<const char*>(E.w[m]);
            for (size_t off = lo + (size_t)lane * kPiece; off < hi; off += 32 * kPiece) {
                const uint32_t n = (uint32_t)min(kPiece, hi - off);
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + off), "r"(n) : "memory");
            }
        }
    }
}

template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- warp helpers
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Reduce 32 values per lane across the warp: afterwards lane l holds the
// warp-wide sum of value l (a reduce-scatter by halving: 31 shuffles).
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16, n = 32; o > 0; o >>= 1, n >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            float send = up ? v[i] : v[i + n / 2];
            float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

// Reduce NV values per lane across the warp (NV a power of two, 2..32):
// halving steps over lane bits 4 .. 5 - log2(NV), then plain sums over the
// remaining low lane bits.  Afterwards lane l holds the warp-wide sum of
// value l >> (5 - log2(NV)).  NV - 1 + 5 - log2(NV) shuffles.
template <int NV>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[NV]) {
    static_assert(NV >= 2 && NV <= 32 && (NV & (NV - 1)) == 0, "NV: power of two in 2..32");
    const int lane = threadIdx.x & 31;
    constexpr int L = NV == 2 ? 1 : NV == 4 ? 2 : NV == 8 ? 3 : NV == 16 ? 4 : 5;
#pragma unroll
    for (int o = 16, n = NV; n > 1; o >>= 1, n >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            float send = up ? v[i] : v[i + n / 2];
            float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float t = v[0];
    if constexpr (L < 5) {
#pragma unroll
        for (int o = 1 << (4 - L); o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    }
    return t;
}

// Reduce 16 values per lane across the warp: afterwards lane l holds the
// warp-wide sum of value (l >> 1) & 15 (halving steps over lane bits 4..1,
// then one exchange over bit 0: 16 shuffles).
__device__ __forceinline__ float warp_reduce_scatter16(float (&v)[16]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16, n = 16; o > 1; o >>= 1, n >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            float send = up ? v[i] : v[i + n / 2];
            float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

}  // namespace moe
