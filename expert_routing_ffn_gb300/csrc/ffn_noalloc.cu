// moe_expert_ffn_noalloc: the expert FFN stage with its scratch memory in a
// fixed, library-owned device array instead of a caller-provided workspace.
//
// Who needs this: code that must not allocate device memory at the moment it
// runs the layer — an engine plugin whose enqueue step is handed only its
// inputs and outputs (the host engine owns the whole memory budget), or a
// decode loop that cannot afford the device-wide synchronisation that
// cudaMalloc/cudaFree imply.  Such callers can still provide inputs and
// outputs; this entry point supplies the rest.
//
// The scratch is a file-scope __device__ array of kScratchBytes (16 MiB).
// Every GPU that loads this library holds it until the process exits.  It
// carries the FFN work plan, the per-CTA partial output rows and an error
// word.  All calls share it and it keeps the previous call's contents, so:
//   - each call clears the error word before its kernels run; the plan and
//     partial rows are fully rewritten before they are read;
//   - calls whose kernels overlap on the GPU (different streams without an
//     ordering between them, or different host threads) race on the array.
//     Order them on one stream, or use moe_expert_ffn with separate
//     workspaces.
// The array's device address is looked up once per CUDA context (the first
// call made while that context is current does it), and remembered under the
// context's unique ID: a context created later, after cudaDeviceReset or by
// the driver API, gets its own lookup.  Make the first call in a context
// outside of any stream capture.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = (size_t)16 << 20;

// In host code this name is a host-side stand-in for the array, not its device
// address: only the address returned by cudaGetSymbolAddress is handed to the
// kernels.
static __device__ __align__(256) unsigned char g_ffn_scratch[kScratchBytes];

std::mutex g_mu;

// One remembered lookup: the context's ID, the array's address in it and the
// SM count of its device.
struct ScratchEntry {
    unsigned long long ctx_id;
    void* ptr;
    int sms;
};
constexpr int kMaxContexts = 64;
ScratchEntry g_entries[kMaxContexts] = {};
int g_n_entries = 0, g_next_slot = 0;

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

// ID of the context current on this thread; 0 if there is none.
cudaError_t current_context_id(unsigned long long* id) {
    *id = 0;
    if (!g_ctx_current || !g_ctx_id) {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa) != cudaSuccess ||
            qa != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
            qb != cudaDriverEntryPointSuccess)
            return cudaErrorNotSupported;
        g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(a);
        g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(b);
    }
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (!ctx) return cudaSuccess;
    return g_ctx_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Device address of g_ffn_scratch in the current context and the SM count of
// the current device (the first call in a context does this set-up).
cudaError_t scratch_for_current_device(void** ptr, int* sms) {
    std::lock_guard<std::mutex> lock(g_mu);
    unsigned long long id = 0;
    cudaError_t e = current_context_id(&id);
    if (e != cudaSuccess) return e;
    if (id != 0)
        for (int i = 0; i < g_n_entries; ++i)
            if (g_entries[i].ctx_id == id) {
                *ptr = g_entries[i].ptr;
                *sms = g_entries[i].sms;
                return cudaSuccess;
            }
    // set-up in this context: the runtime makes the device's primary context
    // current if none is, and loads the module that holds the array
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_ffn_scratch);
    if (e != cudaSuccess) return e;
    int dev = 0, n = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (id == 0) {
        e = current_context_id(&id);
        if (e != cudaSuccess) return e;
    }
    if (id != 0) {
        ScratchEntry& slot = g_entries[g_next_slot];
        slot.ctx_id = id;
        slot.ptr = p;
        slot.sms = n;
        g_next_slot = (g_next_slot + 1) % kMaxContexts;
        if (g_n_entries < kMaxContexts) ++g_n_entries;
    }
    *ptr = p;
    *sms = n;
    return cudaSuccess;
}

struct ScratchLayout {
    size_t err, hdr, segs, seg_first, partial, total;
    int max_segs, max_partial_rows;
};

// Same bounds as the workspace layout, with the actual grid G in place of the
// largest one.
ScratchLayout scratch_layout(const moe_dims& D, int G) {
    ScratchLayout L;
    const size_t T = (size_t)D.T, N = (size_t)D.N;
    const size_t rows_routed = T * (size_t)D.k, rows_shared = T * (size_t)D.n_shared;
    const int rg = moe::gemv_rows(D);
    L.max_segs = (int)(rows_routed / rg + N + (size_t)D.n_shared * (T / rg + 1) + 8);
    L.max_partial_rows = (int)((size_t)rg * G + 2 * (rows_routed + rows_shared) + 16);
    size_t o = 0;
    auto take = [&](size_t b) { size_t at = o; o = moe::align_up(o + b, moe::kAlign); return at; };
    L.err = take(sizeof(moe::DevError));
    L.hdr = take(sizeof(moe::PlanHeader));
    L.segs = take((size_t)L.max_segs * sizeof(moe::Seg));
    L.seg_first = take((N + (size_t)D.n_shared + 1) * 4);
    L.partial = take((size_t)L.max_partial_rows * (size_t)D.d * 4);
    L.total = o;
    return L;
}

}  // namespace

extern "C" moe_status moe_expert_ffn_noalloc(const moe_dims* dims, const void* x,
                                             const void* table, const int32_t* expert_offsets,
                                             const int32_t* perm, float* y_perm, float* y_shared,
                                             int32_t* device_status, void* stream) {
    size_t ws_unused = 0;
    moe_status st = moe_workspace_size(dims, &ws_unused);  // validates dims
    if (st != MOE_OK) return st;
    if (dims->T == 0) return MOE_OK;
    if (!x || !table || !expert_offsets || !perm || !y_perm) return MOE_ERR_INVALID_ARG;
    if (dims->n_shared > 0 && !y_shared) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(table) % 64))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void* base = nullptr;
    int sms = 0;
    if (scratch_for_current_device(&base, &sms) != cudaSuccess) return MOE_ERR_CUDA;
    const int G = moe::gemv_grid_for(dims->d, dims->wtype == MOE_DTYPE_BF16, sms);
    const ScratchLayout L = scratch_layout(*dims, G);
    if (L.total > kScratchBytes) return MOE_ERR_CAPACITY;  // batch too large for 16 MiB
    const bool bf16 = dims->wtype == MOE_DTYPE_BF16;
    moe::DevError* err = moe::ws_at<moe::DevError>(base, L.err);
    if (cudaMemsetAsync(err, 0, sizeof(moe::DevError), s) != cudaSuccess) return MOE_ERR_CUDA;

    moe::PlanArgs pa;
    pa.expert_offsets = expert_offsets; pa.T = dims->T; pa.N = dims->N; pa.n_shared = dims->n_shared;
    pa.I = dims->I; pa.I_shared = dims->I_shared; pa.rg = moe::gemv_rows(*dims); pa.G = G; pa.p_align = 1;
    pa.max_segs = L.max_segs; pa.max_partial_rows = L.max_partial_rows;
    pa.hdr = moe::ws_at<moe::PlanHeader>(base, L.hdr); pa.segs = moe::ws_at<moe::Seg>(base, L.segs);
    pa.seg_first = moe::ws_at<int32_t>(base, L.seg_first); pa.err = err;
    pa.d = dims->d; pa.tc_plan = nullptr;
    if (moe::launch_plan_gemv(pa, s) != cudaSuccess) return MOE_ERR_CUDA;

    moe::GemvParams p;
    p.x = x; p.d = dims->d; p.N = dims->N; p.topk = dims->k; p.NS = moe::gemv_stages(dims->d, bf16);
    p.perm = perm; p.table = static_cast<const moe::ExpertEntry*>(table);
    p.hdr = pa.hdr; p.segs = pa.segs; p.partial = moe::ws_at<float>(base, L.partial); p.err = err;
    p.floe_u = nullptr; p.floe_kept = nullptr; p.floe_list = nullptr; p.I = dims->I; p.words = 0;
    p.up_pass = 0; p.prefetch_shared = 0;
    if (moe::launch_gemv(p, G, bf16, s) != cudaSuccess) return MOE_ERR_CUDA;

    moe::GemvReduceArgs r;
    r.hdr = pa.hdr; r.segs = pa.segs; r.seg_first = pa.seg_first; r.expert_offsets = expert_offsets;
    r.partial = p.partial; r.d = dims->d; r.N = dims->N; r.n_shared = dims->n_shared; r.T = dims->T;
    r.routed_cap = dims->T * dims->k; r.y_perm = y_perm; r.y_shared = y_shared; r.direct = false;
    if (moe::launch_gemv_reduce(r, s) != cudaSuccess) return MOE_ERR_CUDA;

    if (device_status &&
        cudaMemcpyAsync(device_status, err, 2 * sizeof(int32_t), cudaMemcpyDeviceToDevice, s) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
