// Stage 3b, prefill-size batches: the grouped SwiGLU expert FFN on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory), fed
// by TMA.  One persistent launch runs two kinds of tiles:
//   phase 1: for every (expert segment, 128-row tile, 128-channel tile):
//            [gate | up] = X_tile . [Wg_tile ; Wu_tile]^T  (M=128, N=256)
//            epilogue h = SiLU(gate) * up  -> h (bf16)
//   phase 2: for every (segment, 128-row tile, 256-column tile of d):
//            y = h_tile . Wd  (K = I; Wd is [I, d], an MN-major operand)
//            epilogue -> y (fp32, ungated)
// Tiles are numbered phase 1 first, then phase 2; one CTA per tile claims
// numbers in order from a counter, pair c takes c, c + G, ...  A phase-2 tile
// needs the h rows of its (segment, row tile) from every phase-1 channel
// tile: each epilogue warp counts its finished phase-1 tile on that counter
// (after its stores completed), and the producer of a phase-2 tile waits for
// the count before loading h.  Every phase-1 tile is taken before any phase-2
// tile and never waits on another CTA, so every wait ends; the end of phase 1
// and the start of phase 2 overlap instead of a second launch waiting for the
// slowest CTA of the first.
// Shared experts form one segment whose channels are the concatenation of
// all shared experts (so phase 2 sums them, as y_shared requires).
//
// Block: warp 0 issues TMA loads (4-stage ring of 48 KB), warp 1 allocates
// tensor memory and issues the MMAs (one thread), warps 2-5 drain the
// accumulators (one TMEM lane = one tile row per thread).  Accumulators are
// double-buffered (2 x 256 columns) so the epilogue of one tile overlaps the
// MMAs of the next.  The epilogue writes its output through shared memory
// and TMA stores, 32 rows x 128 bytes at a time: a thread owns a row, so
// direct stores would touch 32 cache lines per warp instruction.  Every wait
// is bounded by a clock budget; a timeout sets MOE_ERR_TIMEOUT and all roles
// leave their loops.
#include <cuda.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tma.h"

namespace moe {

constexpr int kTcBM = 128, kTcBN = 256, kTcThreads = 192;
constexpr uint32_t kTcStageA = kTcBM * kTcBK * 2;  // 16 KB
constexpr uint32_t kTcOutBox = 32 * 128;  // one epilogue warp's staging box: 32 rows x 128 bytes
// One CTA per tile: a stage holds A (128 rows) and all of B (256 rows), 4 stages.
// A CTA pair per tile (2-CTA MMA, M = 256): each CTA's stage holds its 128 A
// rows and its half of B, so 6 stages fit in the same shared memory and
// cover 1.5x the load latency at the same MMA rate.
template <bool PAIR>
struct TcCfg {
    static constexpr int kStages = PAIR ? 6 : 4;
    static constexpr uint32_t kStageB = (PAIR ? kTcBN / 2 : kTcBN) * kTcBK * 2;  // 16 / 32 KB
    static constexpr uint32_t kStageBytes = kTcStageA + kStageB;
    static constexpr uint32_t kSmemBytes = kStages * kStageBytes + 4 * kTcOutBox + 1024;  // + alignment slack
};

struct TcParams {
    CUtensorMap map_a_shared;  // phase 1: x [T, d];         phase 2: h_shared [T, ns*Is]
    CUtensorMap map_a_routed;  // phase 1: x_perm [T*k, d];  phase 2: h_routed [T*k, I]
    CUtensorMap map_out_shared;  // phase 1: h_shared (bf16, 64 x 32 boxes); phase 2: y_shared (fp32, 32 x 32)
    CUtensorMap map_out_routed;  // phase 1: h_routed;                       phase 2: y_perm
    const ExpertEntry* table;
    const TcPlan* plan;
    void* out_shared;          // phase 1: h_shared (bf16);  phase 2: y_shared (fp32)
    void* out_routed;          // phase 1: h_routed (bf16);  phase 2: y_perm (fp32)
    long long ld_out_shared, ld_out_routed;  // row strides (elements)
    int d, N, I, I_shared, n_shared;
    DevError* err;
};

// ---------------------------------------------------------------- tiles
struct TcTile {
    int seg, mt, nt;
};

// Tile t of phase `phase` (t counted within the phase); PAIR: 256-row tiles
// (mt counts row pairs).
template <bool PAIR>
__device__ __forceinline__ void tc_tile(const TcPlan& P, int phase, int t, TcTile& out) {
    auto first = [&](const TcSeg& S) {
        return PAIR ? (phase == 1 ? S.tile1p : S.tile2p) : (phase == 1 ? S.tile1 : S.tile2);
    };
    int s = 0;
    while (s + 1 < P.n_seg && first(P.seg[s + 1]) <= t) ++s;
    const TcSeg& S = P.seg[s];
    const int local = t - first(S);
    const int m = PAIR ? S.m_pairs : S.m_tiles;
    out.seg = s;
    out.mt = local % m;
    out.nt = local / m;
}

// Global tile g: phase 1 below the phase-1 tile count, phase 2 after.
template <bool PAIR>
__device__ __forceinline__ int tc_tile_global(const TcPlan& P, int g, TcTile& out) {
    const int n1 = PAIR ? P.n_tiles1p : P.n_tiles1;
    if (g < n1) {
        tc_tile<PAIR>(P, 1, g, out);
        return 1;
    }
    tc_tile<PAIR>(P, 2, g - n1, out);
    return 2;
}

// ---------------------------------------------------------------- CTA pairs
// The 2-CTA forms.  The even CTA of a cluster pair (the leader) issues the
// MMAs, which read both CTAs' shared memory at the same offsets and write
// each CTA's 128 accumulator rows into its own tensor memory; both CTAs'
// stage loads complete on the leader's full barrier; the leader's commits
// arrive on the barrier at the same offset in both CTAs.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// the shared::cluster address of `bar` in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t mapa_rank(const void* bar, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(bar)), "r"(rank));
    return a;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// tile load into this CTA's shared memory, completing on the leader's barrier
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int c0, int c1, uint32_t bar_cl) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(tmap), "r"(c0), "r"(c1), "r"(bar_cl) : "memory");
}
__device__ __forceinline__ void tc_mma_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}
// arrive on `bar` in both CTAs of the pair when the MMAs issued so far are done
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(smem_u32(bar)), "h"((uint16_t)3) : "memory");
}
// the same, on the leader's barrier only
__device__ __forceinline__ void tc_commit_pair_local(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cl) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cl) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// tc_wait with cluster-scope acquire (barriers that the peer CTA signals)
__device__ __forceinline__ bool tc_wait_cl(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           DevError* err, int where, bool honor_abort = true) {
    const long long t0 = clock64();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((i & 63) == 63) {
            if (honor_abort && *abort_flag) return false;
            if (clock64() - t0 > kTcWaitCycles) {
                set_error(err, MOE_ERR_TIMEOUT, where);
                *abort_flag = 1;
                return false;
            }
        }
    }
}
template <bool PAIR>
__device__ __forceinline__ bool tcw(uint64_t* bar, uint32_t parity, volatile int* abort_flag, DevError* err,
                                    int where, bool honor_abort = true) {
    return PAIR ? tc_wait_cl(bar, parity, abort_flag, err, where, honor_abort)
                : tc_wait(bar, parity, abort_flag, err, where, honor_abort);
}

// ---------------------------------------------------------------- phase dependency
// Phase-1 h rows written by other CTAs (TMA stores and plain stores), read by
// this CTA's TMA loads: the writer orders its completed stores before a
// release increment, the reader acquires the count and orders it before its
// async-proxy loads.
__device__ __forceinline__ void dep_signal(int* cnt) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(cnt), "r"(1) : "memory");
}

__device__ __forceinline__ bool dep_wait(const int* cnt, int target, volatile int* abort_flag, DevError* err) {
    const long long t0 = clock64();
    for (uint32_t i = 0;; ++i) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
        if (v >= target) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            return true;
        }
        if ((i & 15) == 15) {
            if (*abort_flag) return false;
            if (clock64() - t0 > kTcWaitCycles) {
                set_error(err, MOE_ERR_TIMEOUT, 7);
                *abort_flag = 1;
                return false;
            }
        }
        __nanosleep(128);
    }
}

// ---------------------------------------------------------------- epilogue stores
// h = SiLU(g) * u = g / (1 + e^-g) * u with the fast exponential and
// division (a few ulp in fp32; h is rounded to bf16).  Very negative g gives
// e^-g = inf and h = -0, the limit.
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g, 1.f + __expf(-g)) * u; }

// 32 consecutive accumulator columns of this thread's TMEM lane, one wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// shared-memory writes of this thread become visible to the TMA (async) proxy
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tma_store_2d(const void* tmap, int c0, int c1, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(tmap), "r"(c0), "r"(c1), "r"(src) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// the staging box may be rewritten: every committed store has read it
__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every committed store has completed
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- kernel
struct TcFusedParams {
    TcParams p1, p2;  // the two phases' tensor maps and outputs
    int* dep;         // per (segment, row tile): phase-1 epilogue warps done (zeroed by the gather)
    int n_dep;        // counters in dep; the last is the tile counter of one-CTA tiles
};

// One CTA per tile: tiles are claimed in order from a global counter, so a
// CTA that drew long tiles takes fewer of the rest.  The producer claims a
// tile and passes its number to the MMA and epilogue warps through a small
// ring in shared memory (kTq slots; a slot is free once all five consumers
// have read it).  A CTA pair keeps the static order (tile stream c takes
// tiles c, c + G, ...), so both CTAs of a pair see the same tiles.
constexpr int kTq = 4;

template <bool PAIR>
__global__ void __launch_bounds__(kTcThreads, 1) ffn_tc_kernel(const __grid_constant__ TcFusedParams fp) {
    using C = TcCfg<PAIR>;
    constexpr int kS = C::kStages;
    grid_dep_wait();  // the plan, x_perm, the zeroed counters: no tensor memory taken before it
    extern __shared__ unsigned char tc_smem_raw[];
    __shared__ __align__(8) uint64_t full[kS], empty[kS], tfull[2], tempty[2], drain;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;
    __shared__ TcPlan plan_s;
    __shared__ int tq[kTq];
    __shared__ __align__(8) uint64_t tq_full[kTq], tq_empty[kTq];

    const TcParams& p = fp.p1;  // fields common to both phases
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t smem_base = (smem_u32(tc_smem_raw) + 1023u) & ~1023u;
    volatile int* abort_flag = &abort_s;
    // PAIR: the cluster is a CTA pair; rank 0 (the leader) issues the MMAs
    const uint32_t rank = PAIR ? cluster_rank() : 0;
    const bool leader = rank == 0;
    const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;  // tile stream of this CTA / pair
    const int n_units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const int pair_rows = PAIR ? 2 * kTcBM : kTcBM;  // rows of a tile
    const int row_off = (int)rank * kTcBM;           // this CTA's rows within the tile
    constexpr int kEpiWarps = PAIR ? 8 : 4;          // epilogue warps per tile (both CTAs)

    for (int i = tid; i < (int)(sizeof(TcPlan) / 4); i += blockDim.x)
        reinterpret_cast<int*>(&plan_s)[i] = reinterpret_cast<const int*>(p.plan)[i];
    if (tid == 0) {
        for (int s = 0; s < kS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps);  // one arrival per epilogue warp (of both CTAs)
        }
        mbar_init(&drain, 1);
        for (int i = 0; i < kTq; ++i) {
            mbar_init(&tq_full[i], 1);
            mbar_init(&tq_empty[i], 1 + kEpiWarps);  // the MMA thread and each epilogue warp
        }
        fence_mbar_init();
        abort_s = 0;
        // the tile counter sits after every (segment, row tile) counter in use
        if (!PAIR && p.plan->n_mt > fp.n_dep - 1) {
            set_error(p.err, MOE_ERR_CAPACITY, p.plan->n_mt);
            abort_s = 1;
        }
    }
    if (warp == 1) {  // tensor memory: 512 columns = two 128x256 fp32 accumulators
        if constexpr (PAIR) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;"
                         ::"r"(smem_u32(&tmem_base_s)));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;"
                         ::"r"(smem_u32(&tmem_base_s)));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // the peer's barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_s;
    const TcPlan& P = plan_s;
    const int d = p.d;
    const int n_tiles = PAIR ? P.n_tiles1p + P.n_tiles2p : P.n_tiles1 + P.n_tiles2;
    // the j-th tile of this CTA, -1 after the last: claimed by the producer
    // (one thread), read by the MMA thread and one lane of each epilogue warp
    auto claim_tile = [&](int j) -> int {
        if constexpr (PAIR) {
            const int g = unit + j * n_units;
            return g < n_tiles ? g : -1;
        } else {
            const int slot = j % kTq;
            if (!tc_wait(&tq_empty[slot], ((j / kTq) & 1) ^ 1, abort_flag, p.err, 7)) return -1;
            int g = atomicAdd(fp.dep + fp.n_dep - 1, 1);
            if (g >= n_tiles) g = -1;
            tq[slot] = g;
            mbar_arrive(&tq_full[slot]);
            return g;
        }
    };
    auto next_tile = [&](int j) -> int {
        if constexpr (PAIR) {
            const int g = unit + j * n_units;
            return g < n_tiles ? g : -1;
        } else {
            const int slot = j % kTq;
            if (!tc_wait(&tq_full[slot], (j / kTq) & 1, abort_flag, p.err, 8)) return -1;
            const int g = tq[slot];
            mbar_arrive(&tq_empty[slot]);
            return g;
        }
    };

    if (warp == 0) {
        // ---------------- TMA producer (each CTA loads its own stages)
        if (lane == 0) {
            int it = 0;
            TcTile tl;
            for (int j = 0; !*abort_flag; ++j) {
                const int g = claim_tile(j);
                if (g < 0) break;
                const int phase = tc_tile_global<PAIR>(P, g, tl);
                const TcSeg& S = P.seg[tl.seg];
                const TcParams& q = phase == 1 ? fp.p1 : fp.p2;
                if (phase == 2 &&
                    !dep_wait(fp.dep + S.mbase + tl.mt, kEpiWarps * S.n1, abort_flag, p.err))
                    break;
                const CUtensorMap* amap = S.shared ? &q.map_a_shared : &q.map_a_routed;
                const int arow = S.row0 + tl.mt * pair_rows + row_off;
                const int nk = phase == 1 ? d / (int)kTcBK
                                          : (S.shared ? p.n_shared * p.I_shared : p.I) / (int)kTcBK;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int st = it % kS;
                    const uint32_t par = ((it / kS) & 1) ^ 1;
                    if (!tcw<PAIR>(&empty[st], par, abort_flag, p.err, 1)) break;
                    const uint32_t a_dst = smem_base + st * C::kStageBytes;
                    const uint32_t b_dst = a_dst + kTcStageA;
                    // the stage's loads complete on the leader's full barrier, which
                    // expects the bytes of both CTAs
                    uint32_t bar = smem_u32(&full[st]);
                    if constexpr (PAIR) bar = mapa_rank(&full[st], 0);
                    if (leader) mbar_arrive_expect_tx(&full[st], (PAIR ? 2 : 1) * C::kStageBytes);
                    auto load = [&](uint32_t dst, const void* tmap, int c0, int c1) {
                        if constexpr (PAIR) tma_load_2d_pair(dst, tmap, c0, c1, bar);
                        else tma_load_2d(dst, tmap, c0, c1, &full[st]);
                    };
                    load(a_dst, amap, kb * kTcBK, arow);
                    if (phase == 1) {
                        int e, nrow;
                        if (S.shared) {
                            const int per = p.I_shared / 128;
                            e = p.N + tl.nt / per;
                            nrow = (tl.nt % per) * 128;
                        } else {
                            e = S.expert;
                            nrow = tl.nt * 128;
                        }
                        const ExpertEntry* E = p.table + e;
                        // B = [gate rows; up rows] (N = 256); a pair splits it by N:
                        // the leader holds the gate rows, the peer the up rows
                        if (!PAIR || leader) load(b_dst, E->tmap[0], kb * kTcBK, nrow);
                        if (!PAIR) load(b_dst + C::kStageB / 2, E->tmap[1], kb * kTcBK, nrow);
                        else if (!leader) load(b_dst, E->tmap[1], kb * kTcBK, nrow);
                    } else {
                        int e, krow;
                        if (S.shared) {
                            const int k0 = kb * kTcBK;
                            e = p.N + k0 / p.I_shared;
                            krow = k0 % p.I_shared;
                        } else {
                            e = S.expert;
                            krow = kb * kTcBK;
                        }
                        const ExpertEntry* E = p.table + e;
                        // B = 256 columns of Wd in 64-column boxes; a pair splits it by N
                        constexpr int kBoxes = (PAIR ? kTcBN / 2 : kTcBN) / 64;
                        const int col0 = tl.nt * kTcBN + (int)rank * (kTcBN / 2) * (PAIR ? 1 : 0);
#pragma unroll
                        for (int j = 0; j < kBoxes; ++j)
                            load(b_dst + j * (64 * kTcBK * 2), E->tmap[2], col0 + j * 64, krow);
                    }
                }
            }
            if constexpr (PAIR) {
                // this CTA's last stages have been consumed by the leader's MMAs
                // (so their loads have landed) before the block may exit
                for (int k = (it > kS ? it - kS : 0); k < it; ++k)
                    (void)tc_wait_cl(&empty[k % kS], (k / kS) & 1, abort_flag, p.err, 2, false);
            } else {
                // wait for the last loads in flight before the block may exit
                for (int k = (it > kS ? it - kS : 0); k < it; ++k)
                    (void)tc_wait(&full[k % kS], (k / kS) & 1, abort_flag, p.err, 2, false);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (the leader of a pair)
        if (lane == 0 && leader) {
            constexpr uint32_t idesc1 = tc_idesc(PAIR ? 2 * kTcBM : kTcBM, kTcBN, 0);
            constexpr uint32_t idesc2 = tc_idesc(PAIR ? 2 * kTcBM : kTcBM, kTcBN, 1);
            int it = 0, local = 0;
            TcTile tl;
            auto mma = [&](uint32_t dt, uint64_t ad, uint64_t bd, uint32_t id, uint32_t acc) {
                if constexpr (PAIR) tc_mma_pair(dt, ad, bd, id, acc);
                else tc_mma(dt, ad, bd, id, acc);
            };
            auto commit = [&](uint64_t* bar) {
                if constexpr (PAIR) tc_commit_pair(bar);
                else tc_commit(bar);
            };
            for (;; ++local) {
                if (*abort_flag) break;
                const int g = next_tile(local);
                if (g < 0) break;
                const int phase = tc_tile_global<PAIR>(P, g, tl);
                const TcSeg& S = P.seg[tl.seg];
                const int ab = local & 1;
                if (!tcw<PAIR>(&tempty[ab], ((local >> 1) & 1) ^ 1, abort_flag, p.err, 3)) break;
                tc_fence_after();
                const uint32_t tmem_d = tmem_base + ab * kTcBN;
                const int nk = phase == 1 ? d / (int)kTcBK
                                          : (S.shared ? p.n_shared * p.I_shared : p.I) / (int)kTcBK;
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int st = it % kS;
                    if (!tcw<PAIR>(&full[st], (it / kS) & 1, abort_flag, p.err, 4)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_base + st * C::kStageBytes;
                    const uint32_t b_addr = a_addr + kTcStageA;
                    if (phase == 1) {
#pragma unroll
                        for (int kk = 0; kk < (int)kTcBK / 16; ++kk)
                            mma(tmem_d, smem_desc(a_addr + kk * 32, 16, 1024), smem_desc(b_addr + kk * 32, 16, 1024),
                                idesc1, (kb | kk) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < (int)kTcBK / 16; ++kk)
                            mma(tmem_d, smem_desc(a_addr + kk * 32, 16, 1024),
                                smem_desc(b_addr + kk * 16 * 128, 64 * kTcBK * 2, 1024), idesc2,
                                (kb | kk) ? 1u : 0u);
                    }
                    commit(&empty[st]);  // frees the stage (in both CTAs) when these MMAs are done
                }
                if (!ok) break;
                commit(&tfull[ab]);      // accumulator ready for the epilogue (of both CTAs)
            }
            // every MMA this thread issued has finished before tensor memory
            // is released
            if constexpr (PAIR) tc_commit_pair_local(&drain);
            else tc_commit(&drain);
            (void)tc_wait(&drain, 0, abort_flag, p.err, 6, false);
        }
    } else {
        // ---------------- epilogue: warps 2..5, thread = accumulator row
        // A warp whose 32 rows all lie in the tile's segment stages each
        // 32-row x 128-byte piece in its shared-memory box (128-byte swizzle:
        // 16-byte chunk j of row i sits at chunk j ^ (i & 7), the layout of
        // the output tensor map) and writes it with one TMA store; the warp
        // that holds a segment's ragged end stores its valid rows directly
        // (the rows after them belong to the next segment).
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t obox = smem_base + kS * C::kStageBytes + quarter * kTcOutBox;
        const uint32_t orow = obox + lane * 128;
        const uint32_t sw = lane & 7;
        // the accumulator's free barrier is the leader's
        uint32_t tempty_cl0 = 0, tempty_cl1 = 0;
        if constexpr (PAIR) {
            tempty_cl0 = mapa_rank(&tempty[0], 0);
            tempty_cl1 = mapa_rank(&tempty[1], 0);
        }
        int local = 0;
        TcTile tl;
        // decisions stay warp-uniform: tcgen05.ld is a whole-warp instruction
        for (;; ++local) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            int g = 0;
            if (lane == 0) g = next_tile(local);
            g = __shfl_sync(0xffffffffu, g, 0);
            if (g < 0) break;
            const int phase = tc_tile_global<PAIR>(P, g, tl);
            const TcSeg& S = P.seg[tl.seg];
            const TcParams& q = phase == 1 ? fp.p1 : fp.p2;
            const int ab = local & 1;
            bool ok = true;
            if (lane == 0) ok = tcw<PAIR>(&tfull[ab], (local >> 1) & 1, abort_flag, p.err, 5);
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + ab * kTcBN;
            const int tile_row = tl.mt * pair_rows + row_off;  // first row of this CTA's part
            const int row_in_seg = tile_row + r;
            const bool valid = row_in_seg < S.rows;
            const bool boxed = tile_row + quarter * 32 + 32 <= S.rows;
            const int box_row = S.row0 + tile_row + quarter * 32;
            const CUtensorMap* omap = S.shared ? &q.map_out_shared : &q.map_out_routed;
            const long long grow = (long long)S.row0 + row_in_seg;
            // rows past the segment's end (the next segment's rows, or the
            // zero fill past the last one) are never stored: a warp holding
            // none of the segment's rows reads nothing, and no thread runs the
            // SiLU on a row it will not store
            const bool any_valid = __any_sync(0xffffffffu, valid);
            if (!any_valid) {
            } else if (phase == 1) {
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(S.shared ? q.out_shared : q.out_routed);
                const long long ld = S.shared ? q.ld_out_shared : q.ld_out_routed;
                __nv_bfloat16* dst = out + grow * ld + (long long)tl.nt * 128;
#pragma unroll 1
                for (int c = 0; c < 128; c += 64) {  // 64 channels = one 128-byte box row
                    if (boxed) {
                        if (lane == 0) tma_store_wait_read();
                        __syncwarp();
                    }
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        float gv[32], uv[32];
                        tmem_ld32(taddr + c + hh * 32, gv);
                        tmem_ld32(taddr + 128 + c + hh * 32, uv);
                        uint32_t w[16];
                        if (valid) {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                w[i] = pack_bf16x2(silu_mul(gv[2 * i], uv[2 * i]), silu_mul(gv[2 * i + 1], uv[2 * i + 1]));
                        }
                        if (boxed) {
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq)
                                st_shared_v4(orow + ((((uint32_t)(hh * 4 + qq)) ^ sw) << 4), w[4 * qq],
                                             w[4 * qq + 1], w[4 * qq + 2], w[4 * qq + 3]);
                        } else if (valid) {
                            uint4* o = reinterpret_cast<uint4*>(dst + c + hh * 32);
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq)
                                o[qq] = make_uint4(w[4 * qq], w[4 * qq + 1], w[4 * qq + 2], w[4 * qq + 3]);
                        }
                    }
                    if (boxed) {
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0) tma_store_2d(omap, tl.nt * 128 + c, box_row, obox);
                    }
                }
            } else {
                float* out = static_cast<float*>(S.shared ? q.out_shared : q.out_routed);
                const long long ld = S.shared ? q.ld_out_shared : q.ld_out_routed;
                float* dst = out + grow * ld + (long long)tl.nt * kTcBN;
#pragma unroll 1
                for (int c = 0; c < kTcBN; c += 32) {  // 32 columns = one 128-byte box row
                    float v[32];
                    tmem_ld32(taddr + c, v);
                    if (boxed) {
                        if (lane == 0) tma_store_wait_read();
                        __syncwarp();
#pragma unroll
                        for (int qq = 0; qq < 8; ++qq)
                            st_shared_v4(orow + (((uint32_t)qq ^ sw) << 4), __float_as_uint(v[4 * qq]),
                                         __float_as_uint(v[4 * qq + 1]), __float_as_uint(v[4 * qq + 2]),
                                         __float_as_uint(v[4 * qq + 3]));
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0) tma_store_2d(omap, tl.nt * kTcBN + c, box_row, obox);
                    } else if (valid) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4*>(dst + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR && !leader) mbar_arrive_remote(ab ? tempty_cl1 : tempty_cl0);
                else mbar_arrive(&tempty[ab]);
            }
            if (phase == 1) {
                // this warp's rows of h are complete in global memory: count
                // them for the phase-2 tiles of this (segment, row tile)
                if (lane == 0) tma_store_wait_all();
                __threadfence();
                __syncwarp();
                if (lane == 0) dep_signal(fp.dep + S.mbase + tl.mt);
            }
        }
        // the block's shared memory stays allocated until these stores have
        // read it, and the output is complete when the grid ends
        if (lane == 0) tma_store_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // a pair: the leader's MMAs (reading the peer's shared memory, writing its
    // tensor memory) are done before either CTA frees or leaves
    if constexpr (PAIR) cluster_sync();
    tc_fence_after();
    if (warp == 1) {
        if constexpr (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;" ::"r"(tmem_base));
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base));
    }
}

// ---------------------------------------------------------------- gather
// x_perm[pos] = x[perm[pos] / k] for the routed rows (bf16, 16-byte copies);
// block 0 also clears the FFN kernel's phase-dependency counters.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ perm,
                                                          const int32_t* __restrict__ expert_offsets,
                                                          int N, int k, int chunks_per_row,
                                                          int rows_cap, uint4* __restrict__ x_perm,
                                                          int* __restrict__ dep, int n_dep) {
    grid_dep_wait();  // the previous kernels' outputs (dependent launch)
    if (blockIdx.x == 0 && dep)
        for (int i = threadIdx.x; i < n_dep; i += blockDim.x) dep[i] = 0;
    const int n_rows = expert_offsets[N];
    for (int pos = blockIdx.x; pos < n_rows && pos < rows_cap; pos += gridDim.x) {
        const int tok = perm[pos] / k;
        for (int c = threadIdx.x; c < chunks_per_row; c += blockDim.x)
            x_perm[(size_t)pos * chunks_per_row + c] = x[(size_t)tok * chunks_per_row + c];
    }
}

// ---------------------------------------------------------------- host
cudaError_t launch_gather_rows(const void* x, const int32_t* perm, const int32_t* expert_offsets, int N,
                               int k, int d, int rows_cap, void* x_perm, cudaStream_t st, int* dep, int n_dep) {
    const int chunks = d / 8;
    const int g_rows = rows_cap < 4096 ? (rows_cap > 0 ? rows_cap : 1) : 4096;
    return launch_pdl(gather_rows_kernel, dim3(g_rows), dim3(256), 0, st, static_cast<const uint4*>(x), perm,
                      expert_offsets, N, k, chunks, rows_cap, static_cast<uint4*>(x_perm), dep, n_dep);
}

// ---------------------------------------------------------------- host
// One CTA per tile, or CTA pairs (clusters of 2) running the 2-CTA MMA:
// -1 chooses by the batch, 0 and 1 force one or the other (tests).  Pairs
// once the routed rows average at least 256 per expert: measured on the same
// GPU, alternating, the FFN stage took 342 against 366 us (DeepSeek-V2-Lite
// shape, 4096 tokens) and 2.52 against 2.57 ms (Qwen2-57B shape); smaller
// segments waste more of a 256-row tile on their ragged end.
static std::atomic<int> g_tc_pairs{-1};

void set_tc_pairs(int mode) { g_tc_pairs.store(mode < 0 ? -1 : (mode > 0 ? 1 : 0)); }

static bool use_tc_pairs(int T, int k, int N) {
    const int m = g_tc_pairs.load();
    if (m >= 0) return m == 1;
    return (long long)T * k >= 256LL * N;
}

template <bool PAIR>
static cudaError_t launch_tc_kernel(const TcFusedParams& fp, int grid, cudaStream_t st) {
    auto kern = ffn_tc_kernel<PAIR>;
    cudaError_t e = allow_max_smem(kern);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = TcCfg<PAIR>::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int n_attr = 1;
    if (PAIR) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n_attr = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    return note_launch(reinterpret_cast<const void*>(kern), kTcThreads, TcCfg<PAIR>::kSmemBytes,
                       cudaLaunchKernelEx(&cfg, kern, fp));
}

// CTA pairs that can be resident at once (every CTA of the persistent grid
// must be: phase-2 tiles wait on phase-1 tiles of other CTAs), at most
// max_ctas / 2; 0 if pairs cannot run.  Cached per device.
static cudaError_t tc_pair_clusters(int max_ctas, int* clusters) {
    static std::mutex mu;
    static int cache[64];
    static bool have[64] = {false};
    *clusters = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        e = allow_max_smem(ffn_tc_kernel<true>);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(max_ctas & ~1);
        cfg.blockDim = dim3(kTcThreads);
        cfg.dynamicSmemBytes = TcCfg<true>::kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, ffn_tc_kernel<true>, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();  // pairs unavailable: one CTA per tile
            n = 0;
        }
        cache[dev] = n;
        have[dev] = true;
    }
    *clusters = cache[dev] < max_ctas / 2 ? cache[dev] : max_ctas / 2;
    return cudaSuccess;
}

cudaError_t launch_tc_ffn(const TcLaunch& a, cudaStream_t st) {
    cudaError_t e = launch_gather_rows(a.x, a.perm, a.expert_offsets, a.N, a.k, a.d, a.rows_cap, a.x_perm, st,
                                       a.dep, a.n_dep);
    if (e != cudaSuccess) return e;

    TcParams p1;
    std::memset(&p1, 0, sizeof(p1));
    if (encode_bf16_2d(&p1.map_a_shared, a.x, a.d, a.T, (uint64_t)a.d * 2, kTcBK, kTcBM) != MOE_OK ||
        encode_bf16_2d(&p1.map_a_routed, a.x_perm, a.d, a.rows_cap, (uint64_t)a.d * 2, kTcBK, kTcBM) != MOE_OK)
        return cudaErrorInvalidValue;
    p1.table = a.table; p1.plan = a.plan;
    p1.out_shared = a.h_shared; p1.out_routed = a.h_routed;
    p1.ld_out_shared = (long long)a.n_shared * a.I_shared; p1.ld_out_routed = a.I;
    // epilogue store maps: 128-byte x 32-row boxes
    const uint64_t hs_cols = (uint64_t)a.n_shared * a.I_shared;
    if (a.n_shared > 0 &&
        encode_bf16_2d(&p1.map_out_shared, a.h_shared, hs_cols, a.T, hs_cols * 2, 64, 32) != MOE_OK)
        return cudaErrorInvalidValue;
    if (encode_bf16_2d(&p1.map_out_routed, a.h_routed, a.I, a.rows_cap, (uint64_t)a.I * 2, 64, 32) != MOE_OK)
        return cudaErrorInvalidValue;
    p1.d = a.d; p1.N = a.N; p1.I = a.I; p1.I_shared = a.I_shared; p1.n_shared = a.n_shared; p1.err = a.err;

    TcParams p2 = p1;
    if (a.n_shared > 0 &&
        encode_bf16_2d(&p2.map_a_shared, a.h_shared, hs_cols, a.T, hs_cols * 2, kTcBK, kTcBM) != MOE_OK)
        return cudaErrorInvalidValue;
    if (encode_bf16_2d(&p2.map_a_routed, a.h_routed, a.I, a.rows_cap, (uint64_t)a.I * 2, kTcBK, kTcBM) != MOE_OK)
        return cudaErrorInvalidValue;
    p2.out_shared = a.y_shared; p2.out_routed = a.y_perm;
    if (a.n_shared > 0 &&
        encode_f32_2d(&p2.map_out_shared, a.y_shared, a.d, a.T, (uint64_t)a.d * 4, 32, 32) != MOE_OK)
        return cudaErrorInvalidValue;
    if (encode_f32_2d(&p2.map_out_routed, a.y_perm, a.d, a.rows_cap, (uint64_t)a.d * 4, 32, 32) != MOE_OK)
        return cudaErrorInvalidValue;
    p2.ld_out_shared = a.d; p2.ld_out_routed = a.d;

    TcFusedParams fp;
    fp.p1 = p1;
    fp.p2 = p2;
    fp.dep = a.dep;
    fp.n_dep = a.n_dep;
    int clusters = 0;
    if (use_tc_pairs(a.T, a.k, a.N)) {
        e = tc_pair_clusters(a.grid, &clusters);
        if (e != cudaSuccess) return e;
    }
    if (clusters > 0) return launch_tc_kernel<true>(fp, 2 * clusters, st);
    return launch_tc_kernel<false>(fp, a.grid, st);
}

}  // namespace moe
