// TMA tensor-map encoding through the driver entry point (the library does not
// link libcuda; the driver is found at run time like the rest of the CUDA
// runtime).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "tma.h"

namespace moe {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

moe_status encode_2d(void* out128, CUtensorMapDataType type, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return MOE_ERR_CUDA;
    if ((reinterpret_cast<uintptr_t>(base) & 15u) || (row_stride_bytes & 15u)) return MOE_ERR_INVALID_ARG;
    CUtensorMap m;
    std::memset(&m, 0, sizeof(m));
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(&m, type, 2, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return MOE_ERR_INVALID_ARG;
    std::memcpy(out128, &m, sizeof(m));
    return MOE_OK;
}

}  // namespace

moe_status encode_bf16_2d(void* out128, const void* base, uint64_t inner, uint64_t outer,
                          uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    return encode_2d(out128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, outer, row_stride_bytes, box_inner,
                     box_outer);
}

moe_status encode_f32_2d(void* out128, const void* base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    return encode_2d(out128, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, inner, outer, row_stride_bytes, box_inner,
                     box_outer);
}

moe_status encode_expert_tmaps(ExpertEntry& E, int d) {
    // gate / up: K-major tiles of 128 channels x 64 hidden values
    for (int m = 0; m < 2; ++m)
        if (moe_status s = encode_bf16_2d(E.tmap[m], E.w[m], (uint64_t)d, (uint64_t)E.I,
                                          (uint64_t)d * 2, kTcBK, 128);
            s != MOE_OK)
            return s;
    // down: MN-major tiles of 64 hidden values (contiguous) x 64 channels (K)
    if (moe_status s = encode_bf16_2d(E.tmap[2], E.w[2], (uint64_t)d, (uint64_t)E.I, (uint64_t)d * 2, 64, kTcBK);
        s != MOE_OK)
        return s;
    // decode path: all three in 16-row boxes of 64 values
    for (int m = 0; m < 3; ++m)
        if (moe_status s = encode_bf16_2d(E.tmap_dec[m], E.w[m], (uint64_t)d, (uint64_t)E.I,
                                          (uint64_t)d * 2, kTcBK, 16);
            s != MOE_OK)
            return s;
    return MOE_OK;
}

}  // namespace moe
