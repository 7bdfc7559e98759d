// Stage 3b for a batch of one token: the SwiGLU expert FFN as an
// HBM-streaming GEMV with one channel per warp.
//
// y = sum_i SiLU(x . Wg[i]) (x . Wu[i]) Wd[i, :]  (FloE method §1 with the
// identity mask; weights channel-major [I, d], so channel i's gate, up and
// down rows are three contiguous d-vectors).
//
// With one token every segment of the GEMV plan has one row, and the
// per-stage block reduction of ffn_gemv.cu (a warp reduce-scatter, a block
// barrier, a cross-warp sum) costs more instructions than the weights' own
// multiply-adds.  Here each warp owns whole channels: the two dot products
// are warp all-reduces and no block barrier runs per channel.
//
// Work split: the GEMV plan's (the channels of all segments cut into G
// ranges, one per CTA; one partial output row per CTA and segment piece), so
// the plan, the partial rows and their reduction are those of ffn_gemv.cu.
// Inside a CTA, warp w takes channels w, w + kW1Warps, ... of each segment
// piece and streams them through a private ring of kW1Slots slots (gate, up
// and down row of one channel per slot) that its lane 0 fills with 1-D bulk
// copies (the TMA engine), evict-first in L2.  Lane l owns the 16-byte chunks
// l, l + 32, ... of d, so shared-memory reads are conflict-free, and keeps x
// and its output columns in registers.  At the end of a segment piece the
// warps' rows are added in warp order through shared memory, one chunk per
// lane at a time, and written as the CTA's partial row.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kW1Warps = 4;
constexpr int kW1Threads = 32 * kW1Warps;
constexpr int kW1Slots = 2;

__host__ __device__ inline size_t gemv1_smem_bytes(int d) {
    // ring [warp][slot][3 rows][d] bf16, then two reduction buffers of
    // [warp][2 halves][32 lanes] float4
    return (size_t)kW1Warps * kW1Slots * 3 * d * 2 + 2 * (size_t)kW1Warps * 2 * 32 * 16;
}

// Lane 0's copy issuer: walks the warp's channels in the order it consumes
// them (segment pieces of the CTA's range, channels w, w + kW1Warps, ...).
struct W1Producer {
    const Seg* segs;
    const ExpertEntry* table;
    int seg, n_seg, lo, hi, w;  // current segment, CTA range [lo, hi) of the global channel list
    int c;                      // next local channel of segment `seg` to issue
    int c_start, c_end;         // local bounds of the piece of `seg`
    int cached;
    const char* wp[3];
    size_t row_bytes;
    uint64_t policy;

    __device__ __forceinline__ void load_seg() {
        const Seg S = segs[seg];
        const ExpertEntry& E = table[S.expert];
#pragma unroll
        for (int m = 0; m < 3; ++m) wp[m] = static_cast<const char*>(E.w[m]);
        c_start = max(lo, S.ch_start) - S.ch_start;
        c_end = min(hi, S.ch_start + S.I) - S.ch_start;
        c = c_start + w;
        cached = seg;
    }
    // advance to the next channel to issue; false when the range is done
    __device__ __forceinline__ bool next() {
        while (seg < n_seg) {
            if (cached != seg) {
                if (segs[seg].ch_start >= hi) { seg = n_seg; return false; }
                load_seg();
            }
            if (c < c_end) return true;
            ++seg;
        }
        return false;
    }
    __device__ __forceinline__ void issue(unsigned char* slot, uint64_t* bar) {
        const uint32_t rb = (uint32_t)row_bytes;
        mbar_arrive_expect_tx(bar, 3 * rb);
#pragma unroll
        for (int m = 0; m < 3; ++m)
            bulk_g2s(slot + m * row_bytes, wp[m] + (size_t)c * row_bytes, rb, bar, policy);
        c += kW1Warps;
    }
};

template <int DV>  // 16-byte chunks of d per lane (d = 256 * DV)
__global__ void __launch_bounds__(kW1Threads, 2) ffn_gemv1_kernel(GemvParams p) {
    extern __shared__ __align__(128) unsigned char smem1[];
    __shared__ __align__(8) uint64_t full[kW1Warps][kW1Slots];
    constexpr int d = 256 * DV;
    constexpr size_t row_bytes = (size_t)d * 2;
    constexpr size_t slot_bytes = 3 * row_bytes;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (w == 0 && p.prefetch_shared > 0)
        l2_prefetch_shared_experts(p.table, p.N, p.prefetch_shared, d, 2, blockIdx.x, gridDim.x, lane);
    grid_dep_wait();  // the plan comes from the previous kernels
    const PlanHeader hdr = *p.hdr;
    const int cta = blockIdx.x;
    if (cta >= hdr.G) return;
    const int lo = cta * hdr.P, hi = min(lo + hdr.P, hdr.total_ch);
    if (lo >= hi || hdr.n_seg <= 0) return;
    int s_lo = 0, s_hi = hdr.n_seg - 1;  // the segment holding channel lo
    while (s_lo < s_hi) {
        const int mid = (s_lo + s_hi + 1) >> 1;
        if (p.segs[mid].ch_start <= lo) s_lo = mid; else s_hi = mid - 1;
    }
    const int seg0 = s_lo;

    unsigned char* ring = smem1 + (size_t)w * kW1Slots * slot_bytes;
    float4* red = reinterpret_cast<float4*>(smem1 + (size_t)kW1Warps * kW1Slots * slot_bytes);
    uint64_t* bars = full[w];

    W1Producer prod;
    int issued = 0;
    if (lane == 0) {
        for (int s = 0; s < kW1Slots; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
        prod.segs = p.segs; prod.table = p.table; prod.seg = seg0; prod.n_seg = hdr.n_seg;
        prod.lo = lo; prod.hi = hi; prod.w = w; prod.cached = -1; prod.row_bytes = row_bytes;
        prod.policy = l2_evict_first_policy();
        for (int s = 0; s < kW1Slots && prod.next(); ++s) {
            prod.issue(ring + s * slot_bytes, &bars[s]);
            ++issued;
        }
    }
    __syncwarp();

    // x (the batch's one token) in registers: chunk j of this lane holds
    // elements 8 (lane + 32 j) .. + 7
    float xr[DV][8];
    {
        const uint4* xv = static_cast<const uint4*>(p.x);
#pragma unroll
        for (int j = 0; j < DV; ++j) unpack16(xv[lane + 32 * j], xr[j], (__nv_bfloat16*)nullptr);
    }

    bool abort = false;
    int k = 0;          // channels of this warp passed (consumed, or skipped after a timeout)
    int drain_from = 0;  // first channel whose copy may still be in flight at the end
    int rbuf = 0;
    for (int seg = seg0; seg < hdr.n_seg; ++seg) {
        const Seg S = p.segs[seg];
        if (S.ch_start >= hi) break;
        const int c_lo = max(lo, S.ch_start) - S.ch_start, c_hi = min(hi, S.ch_start + S.I) - S.ch_start;
        float acc[DV][8];
#pragma unroll
        for (int j = 0; j < DV; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
        for (int c = c_lo + w; c < c_hi; c += kW1Warps, ++k) {
            const int s = k % kW1Slots;
            if (!abort) {
                // every lane waits (each needs the acquire of the copies' bytes);
                // the warp gives up together if any lane's wait ran out
                const bool ok = mbar_wait(&bars[s], (uint32_t)((k / kW1Slots) & 1));
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) set_error(p.err, MOE_ERR_TIMEOUT, cta);
                    abort = true;
                    drain_from = k;
                }
            }
            if (abort) continue;
            const unsigned char* slot = ring + s * slot_bytes;
            const uint4* gr = reinterpret_cast<const uint4*>(slot);
            const uint4* ur = reinterpret_cast<const uint4*>(slot + row_bytes);
            const uint4* dr = reinterpret_cast<const uint4*>(slot + 2 * row_bytes);
            float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
            for (int j = 0; j < DV; ++j) {
                float wg[8], wu[8];
                unpack16(gr[lane + 32 * j], wg, (__nv_bfloat16*)nullptr);
                unpack16(ur[lane + 32 * j], wu, (__nv_bfloat16*)nullptr);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    fma2(g0, g1, wg[e], wg[e + 1], xr[j][e], xr[j][e + 1]);
                    fma2(u0, u1, wu[e], wu[e + 1], xr[j][e], xr[j][e + 1]);
                }
            }
            float g = g0 + g1, u = u0 + u1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                g += __shfl_xor_sync(0xffffffffu, g, o);
                u += __shfl_xor_sync(0xffffffffu, u, o);
            }
            const float h = g / (1.f + expf(-g)) * u;
#pragma unroll
            for (int j = 0; j < DV; ++j) {
                float wd[8];
                unpack16(dr[lane + 32 * j], wd, (__nv_bfloat16*)nullptr);
#pragma unroll
                for (int e = 0; e < 8; e += 2) fma2(acc[j][e], acc[j][e + 1], h, h, wd[e], wd[e + 1]);
            }
            __syncwarp();  // every lane has read the slot
            if (lane == 0 && prod.next()) {
                prod.issue(ring + s * slot_bytes, &bars[s]);
                ++issued;
            }
        }
        // the CTA's partial row of this segment: the warps' rows added in
        // warp order, one chunk per lane at a time (double-buffered)
        float* dst = p.partial + (size_t)(S.pbase + (cta - S.c0)) * d;
#pragma unroll
        for (int j = 0; j < DV; ++j) {
            float4* b = red + (size_t)rbuf * kW1Warps * 64;
            b[(w * 2 + 0) * 32 + lane] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
            b[(w * 2 + 1) * 32 + lane] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
            __syncthreads();
            if (tid < 64) {
                const int half = tid >> 5, l = tid & 31;
                float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int v = 0; v < kW1Warps; ++v) add4(y, b[(v * 2 + half) * 32 + l]);
                *reinterpret_cast<float4*>(dst + (size_t)(l + 32 * j) * 8 + half * 4) = y;
            }
            rbuf ^= 1;
        }
        __syncthreads();  // both reduction buffers free for the next piece
    }
    // copies still in flight (after a timeout): wait for them, bounded,
    // before the CTA's shared memory is released
    if (lane == 0)
        for (int q = abort ? drain_from : k; q < issued; ++q)
            (void)mbar_wait(&bars[q % kW1Slots], (uint32_t)((q / kW1Slots) & 1));
}

bool gemv1_usable(int T, int d, bool bf16, bool floe) {
    return T == 1 && bf16 && !floe && (d == 1536 || d == 2048);
}

cudaError_t launch_gemv1(const GemvParams& p, int G, cudaStream_t st) {
    const size_t smem = gemv1_smem_bytes(p.d);
    auto run = [&](auto kernel) {
        cudaError_t e = allow_max_smem(kernel);
        if (e != cudaSuccess) return e;
        e = launch_pdl(kernel, dim3(G), dim3(kW1Threads), smem, st, p);
        return note_launch(reinterpret_cast<const void*>(kernel), kW1Threads, smem, e);
    };
    if (p.d == 2048) return run(ffn_gemv1_kernel<8>);
    if (p.d == 1536) return run(ffn_gemv1_kernel<6>);
    return cudaErrorInvalidValue;
}

}  // namespace moe
