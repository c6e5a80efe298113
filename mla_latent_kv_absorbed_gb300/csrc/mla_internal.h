// Shared between the host shim and the kernels: status codes, the plan word
// layout and the launch parameter blocks.
#pragma once

#include <cstddef>
#include <cstdint>

#include "mla_decode.h"

namespace mla {

constexpr int kLatent = 512;       // kv_lora_rank
constexpr int kRope = 64;          // qk_rope_head_dim
constexpr int kRow = kLatent + kRope;  // 576 bf16 per cache row

// ---- plan words --------------------------------------------------------
constexpr int32_t kPlanMagic = 0x4D4C4131;
constexpr int32_t kPlanVersion = 1;
constexpr int kHeaderWords = 16;
enum PlanHeader : int {
  kHMagic = 0, kHVersion, kHBatch, kHHeads, kHVariant, kHTile, kHWorkers, kHCap /* load budget per worker, tokens */,
  kHItems, kHPartials, kHMerges, kHHeadGroups, kHCtasPerWorker, kHTotalWords, kHNumSms,
  kHReserved
};
constexpr int kVariantSwab = 1;  // H in {16, 32}: one CTA per worker, 64-token tiles
constexpr int kVariantPair = 2;  // H in 48..128: a 2-CTA cluster per worker, 64-token tiles
// plan cost of one work item beyond its tiles, in tokens: the item's epilogue
// and the pipeline refill behind it (measured: about half a tile for the
// one-CTA kernel, about four tiles for the two-CTA kernel, whose epilogue
// writes 128 heads x 256 dims per CTA while the next item's softmax waits)
constexpr int item_overhead_tokens(int variant) { return variant == kVariantPair ? 256 : 32; }
constexpr int kMinPieceTokens = 64;       // no cut piece is shorter
constexpr int kCapStepTokens = 8;         // the budget grows in these steps until the fill fits
constexpr size_t kWsHeaderBytes = 256;

// offsets of the plan arrays, from the header
inline int plan_wptr_off(const int32_t* h) { (void)h; return kHeaderWords; }
inline int plan_items_off(const int32_t* h) { return kHeaderWords + h[kHWorkers] + 1; }
inline int plan_merge_off(const int32_t* h) { return plan_items_off(h) + 4 * h[kHItems]; }

// ---- kernel parameters -------------------------------------------------
struct DecodeParams {
  const int32_t* plan;        // device plan words
  const int32_t* kv_indptr;   // device [B+1]
  const int32_t* kv_indices;  // device [nnz]
  const uint16_t* q_nope;     // device bf16 [B, H, 512] (read directly by the pair kernels)
  const uint16_t* q_rope;     // device bf16 [B, H, 64] (read directly by the FP8 pair kernel)
  const uint8_t* kv_cache;    // device [num_slots, 576] bf16 rows (for whole-row L2 prefetch)
  void* out;                  // [B, H, 512] fp32 or bf16
  float* lse;                 // [B, H] or null
  float* part_o;              // [P, H, 512]
  float* part_lse;            // [P, H]
  int* status;                // workspace status word
  long long num_slots;
  int batch;
  int heads;
  int out_bf16;
  int items_off;
  int num_workers;
  float scale_log2;           // sm_scale * log2(e)
  int q_len;                  // queries per request (rows = q_len x heads per query); <= 1: one
  int plan_cap_words;         // > 0: a device-only plan (graph replays) of at most this many words, checked
                              // and clamped by the kernels; 0: a plan the host has checked
  int max_partials;           // partial states the workspace holds; an item naming another writes nothing
  const unsigned long long* tree_masks;   // q_len > 1: per request and draft [B, q_len] the ancestor-or-self
                                          // bits of a draft tree, or null for a chain of drafts
};

struct MergeParams {
  const float* part_o;
  const float* part_lse;
  const int32_t* list;        // plan merge entries (b, p0, p1) x n, or null
  const int32_t* indptr;      // CSR partial ranges [B+1] (when list is null)
  int n_entries;
  int heads;
  void* out;
  int out_bf16;
  float* lse;
  const int32_t* plan;        // device-only plan: entries, list and bounds are read from it (list is null)
  int plan_cap_words;
  int batch;                  // requests the buffers hold
  int max_partials;
  int workers;                // the decode launch's workers (a device-only plan must match)
  int* status;                // workspace status word (device-only plan), or null
};

// Per-head product C[b, h, :] = A[b, h, 0:K] . W[h] (the query absorption and
// the output projection); A and W are read through tensor maps.
struct HeadGemmParams {
  void* out;                  // [rows, heads, N] bf16 or fp32
  int* status;                // status word (MLA_ERR_TIMEOUT), or null
  int rows;                   // B
  int heads;                  // H
};

// Cache append: rows [rows, 576] bf16 to kv_cache[slots[r]].
struct AppendParams {
  void* kv_cache;             // [num_slots, 576] bf16
  const void* src;            // [rows, 576] bf16
  const int32_t* slots;       // [rows]
  int* status;                // status word, or null
  long long num_slots;
  int rows;
};

// FP8 cache decode: the prep kernel's outputs, read by the decode kernel.
struct Fp8Params {
  const uint8_t* img;         // [B] query images (4H x 288 bytes each)
  const float* fac;           // [B, H] per-head factors 2^-a
  float kv_scale;             // cache value = E4M3 code value x kv_scale
};

// FP8 query prep: bf16 q_nope / q_rope -> query images and factors.
struct Fp8PrepParams {
  const uint16_t* q_nope;     // [B, H, 512] bf16
  const uint16_t* q_rope;     // [B, H, 64] bf16
  uint8_t* img;               // [B] images
  float* fac;                 // [B, H]
  int rows;                   // B * H
};

// FP8 cache append: rows [rows, 576] bf16 -> E4M3 codes of value / kv_scale.
struct AppendFp8Params {
  uint8_t* kv_cache;          // [num_slots, 576] E4M3
  const uint16_t* src;        // [rows, 576] bf16
  const int32_t* slots;       // [rows]
  int* status;                // status word, or null
  long long num_slots;
  int rows;
  float kv_scale;
};

}  // namespace mla
