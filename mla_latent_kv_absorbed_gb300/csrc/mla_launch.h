// Launchers of the device kernels, called by the C-ABI shim (mla_api.cpp).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "mla_internal.h"

namespace mla {

// Raises a kernel's dynamic shared-memory limit to `bytes` in the current
// context (once per kernel and context; later calls return at once).  false:
// the CUDA call failed.
bool set_smem_limit(const void* func, int bytes);

// SM count of the current device (cached per device), or 0 on an error.
int device_sm_count();

// Decode kernel for H in {16, 32}; grid = plan workers.  tm_kv: bf16 rows, box
// {64, 1}, 128-byte swizzle; tm_kr: the same rows, box {32, 1}, 64-byte swizzle
// (the rope halves).
int launch_swab(int heads, const CUtensorMap& tm_kv, const CUtensorMap& tm_kr, const CUtensorMap& tm_qn,
                const CUtensorMap& tm_qr, const DecodeParams& p, int grid, cudaStream_t stream);

// Decode kernel for H in 48..128 (a two-CTA cluster per worker); grid = 2 * workers.
int launch_pair(int heads, const CUtensorMap& tm_kv, const CUtensorMap& tm_kv_rope,
                const CUtensorMap& tm_qr, const DecodeParams& p, int workers, cudaStream_t stream);

// LSE merge of partial states; one block per (entry, head).  max_pieces: the
// most partials an entry has (sizes the block), or 0 when unknown.
int launch_merge(const MergeParams& p, int entries, int max_pieces, cudaStream_t stream);

// Query absorption q_nope[b,h,:] = q_pre[b,h,0:128] . w_kc[h] (128 x 512), bf16 out.
// tm_a over q_pre as [B, H*128] (box 64 x 128), tm_w over w_kc as [H*128, 512] (box 64 x 64).
int launch_absorb(const CUtensorMap& tm_a, const CUtensorMap& tm_w, const HeadGemmParams& p, cudaStream_t stream);

// Output projection out[b,h,:] = o_lat[b,h,0:512] . w_vc[h] (512 x 128), bf16 or fp32 out.
// tm_a over o_lat as [B, H*512] (box 64 x 128), tm_w over w_vc as [H*512, 128] (box 64 x 64).
int launch_project(const CUtensorMap& tm_a, const CUtensorMap& tm_w, const HeadGemmParams& p, int out_bf16,
                   cudaStream_t stream);

// Merge of two states per row ([rows, 512] fp32 + [rows] lse each).
int launch_merge_two(const float* o_a, const float* l_a, const float* o_b, const float* l_b, void* out, int out_bf16,
                     float* lse, long long rows, cudaStream_t stream);

// Ancestor-or-self masks of B draft trees of W <= 64 drafts (parents [B, W]
// int32 -> masks [B, W] uint64); a bad parent records MLA_ERR_TREE in status.
int launch_tree_masks(const int32_t* parents, int batch, int width, unsigned long long* masks, int* status,
                      cudaStream_t stream);

// Cache append of a step's new rows.
int launch_append(const AppendParams& p, cudaStream_t stream);

// FP8-cache decode for H in {16, 32}: the query prep kernel, then the decode
// kernel as its programmatic dependent; grid = plan workers.  tm_lat: uint8
// [num_slots, 576], box {128, 1}, 128-B swizzle; tm_rope: box {32, 1}, 32-B swizzle.
int launch_swab8(int heads, const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const DecodeParams& p,
                 const Fp8Params& p8, const Fp8PrepParams& pp, int grid, cudaStream_t stream);

// FP8-cache decode for H in 48..128 (a two-CTA cluster per worker, the query
// split in-kernel); grid = 2 * workers.  tm_lat: uint8 [num_slots, 576], box
// {128, 1}, 128-byte swizzle; tm_rope: box {32, 1}, 32-byte swizzle.
int launch_pair8(int heads, const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const DecodeParams& p,
                 float kv_scale, int workers, cudaStream_t stream);

// Bytes of one request's query image for the FP8 decode.
size_t fp8_image_bytes(int heads);

// FP8 cache append (quantises bf16 rows).
int launch_append_fp8(const AppendFp8Params& p, cudaStream_t stream);

}  // namespace mla
