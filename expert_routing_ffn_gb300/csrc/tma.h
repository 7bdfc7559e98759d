// Host-side encoding of TMA tensor maps for the expert weights.
#pragma once

#include "common.cuh"

namespace moe {

// Encode the tensor maps of one expert (bf16 [I, d] gate/up/down) into E.
moe_status encode_expert_tmaps(ExpertEntry& E, int d);

}  // namespace moe
