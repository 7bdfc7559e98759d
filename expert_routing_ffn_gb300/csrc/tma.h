// Host-side encoding of TMA tensor maps (bf16 or fp32, 2-D, 128-byte swizzle).
#pragma once

#include "common.cuh"

namespace moe {

constexpr uint32_t kTcBK = 64;  // K extent of one tensor-core pipeline stage (128 bytes of bf16)

// A 2-D bf16 tensor [outer][inner] with the given row stride, read in boxes
// of box_outer rows x box_inner values into 128-byte-swizzled shared memory.
moe_status encode_bf16_2d(void* out128, const void* base, uint64_t inner, uint64_t outer,
                          uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

// The same for a 2-D fp32 tensor (boxes of at most 32 values: 128 bytes).
moe_status encode_f32_2d(void* out128, const void* base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

// The three tensor maps of one expert (bf16 [I, d] gate/up/down) into E.
moe_status encode_expert_tmaps(ExpertEntry& E, int d);

}  // namespace moe
