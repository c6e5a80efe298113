// Launchers of the device kernels, called by the C-ABI shim (mla_api.cpp).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "mla_internal.h"

namespace mla {

// Decode kernel for H in {16, 32}; grid = plan workers.
int launch_swab(int heads, const CUtensorMap& tm_kv, const CUtensorMap& tm_qn,
                const CUtensorMap& tm_qr, const DecodeParams& p, int grid, cudaStream_t stream);

// Decode kernel for H in 48..128 (a two-CTA cluster per worker); grid = 2 * workers.
int launch_pair(int heads, const CUtensorMap& tm_kv, const CUtensorMap& tm_kv_rope,
                const CUtensorMap& tm_qr, const DecodeParams& p, int workers, cudaStream_t stream);

// LSE merge of partial states; one block per (entry, head).  max_pieces: the
// most partials an entry has (sizes the block), or 0 when unknown.
int launch_merge(const MergeParams& p, int entries, int max_pieces, cudaStream_t stream);

}  // namespace mla
