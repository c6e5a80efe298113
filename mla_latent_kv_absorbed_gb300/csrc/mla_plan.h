// Host plan builder (see mla_plan.cpp for the rule).
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "mla_internal.h"

namespace mla {

// Returns the variant for H (kVariantSwab / kVariantPair) and its tile size
// and CTAs per worker, or 0 when H is not supported.
int variant_for_heads(int H, int* tile, int* ctas_per_worker);

// Builds the plan words for a host kv_indptr[B+1] (already validated).
int build_plan(const int32_t* indptr, int B, int H, int num_sms, std::vector<int32_t>& words,
               size_t* workspace_bytes);

size_t ws_part_o_offset();
size_t ws_part_lse_offset(const int32_t* header);
// Workspace bytes mla_decode_run needs for a plan: status header, fp32
// partial states [P,H,512] and their LSEs [P,H].
size_t ws_needed_bytes(const int32_t* header);

}  // namespace mla
