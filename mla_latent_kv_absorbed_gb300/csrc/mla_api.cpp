// The C ABI of libmla_decode.so (declared in include/mla_decode.h): argument
// checks, the host plan, TMA descriptor encoding and kernel dispatch.  Nothing
// here allocates device memory or synchronises except mla_check_errors.
#include <algorithm>
#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "mla_launch.h"
#include "mla_plan.h"

using namespace mla;

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] array, box {box_cols, box_rows},
// 128-byte swizzle (64-byte for boxes 64 bytes wide).
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool plan_header_ok(const int32_t* h) {
  if (!h || h[kHMagic] != kPlanMagic || h[kHVersion] != kPlanVersion) return false;
  int T = 0, cpw = 0;
  const int v = variant_for_heads(h[kHHeads], &T, &cpw);
  if (!v || v != h[kHVariant] || T != h[kHTile] || cpw != h[kHCtasPerWorker]) return false;
  if (h[kHBatch] < 0 || h[kHWorkers] < 1 || h[kHItems] < 0 || h[kHPartials] < 0 || h[kHMerges] < 0)
    return false;
  const long long words = kHeaderWords + (static_cast<long long>(h[kHWorkers]) + 1) +
                          4ll * h[kHItems] + 3ll * h[kHMerges];
  return words == h[kHTotalWords];
}

}  // namespace

extern "C" {

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_INDEX_OOB: return "MLA_ERR_INDEX_OOB";
    case MLA_ERR_PLAN_MISMATCH: return "MLA_ERR_PLAN_MISMATCH";
    case MLA_ERR_TREE: return "MLA_ERR_TREE";
    default: return "MLA_ERR_UNKNOWN";
  }
}

int mla_abi_version(void) { return 1; }

int mla_decode_plan(const int32_t* kv_indptr, int32_t batch, int32_t num_heads, int32_t num_sms,
                    int32_t* plan, size_t plan_words, size_t* plan_words_needed,
                    size_t* workspace_bytes) {
  if (batch < 0 || !kv_indptr) return MLA_ERR_INVALID_ARG;
  if (kv_indptr[0] != 0) return MLA_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b)
    if (kv_indptr[b + 1] < kv_indptr[b]) return MLA_ERR_INVALID_ARG;
  int T = 0, cpw = 0;
  if (!variant_for_heads(num_heads, &T, &cpw)) return MLA_ERR_UNSUPPORTED;
  if (num_sms < 0) return MLA_ERR_INVALID_ARG;
  if (num_sms == 0) {
    // the SM count of the current device (cached per device; plans may be
    // built from several host threads at once)
    num_sms = device_sm_count();
    if (num_sms < 1) return MLA_ERR_CUDA;
  }
  std::vector<int32_t> words;
  size_t ws = 0;
  const int st = build_plan(kv_indptr, batch, num_heads, num_sms, words, &ws);
  if (st != MLA_OK) return st;
  if (plan_words_needed) *plan_words_needed = words.size();
  if (workspace_bytes) *workspace_bytes = ws;
  if (!plan) return MLA_OK;
  if (plan_words < words.size()) return MLA_ERR_WORKSPACE;
  std::memcpy(plan, words.data(), words.size() * sizeof(int32_t));
  return MLA_OK;
}

namespace {

int check_run_args(const int32_t* plan_host, const int32_t* plan_dev, int32_t out_dtype, void* workspace,
                   size_t workspace_bytes) {
  if (!plan_header_ok(plan_host) || !plan_dev) return MLA_ERR_INVALID_ARG;
  if (out_dtype != 0 && out_dtype != 1) return MLA_ERR_UNSUPPORTED;
  const size_t need = ws_needed_bytes(plan_host);
  if (!workspace || !aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < need) return MLA_ERR_WORKSPACE;
  return MLA_OK;
}

}  // namespace

namespace {
int attend_impl(const int32_t* plan_host, const int32_t* plan_dev, int32_t q_len, const void* q_nope,
                const void* q_rope, const void* kv_cache, int64_t num_slots, const int32_t* kv_indptr,
                const int32_t* kv_indices, float sm_scale, void* out, int32_t out_dtype, float* lse,
                void* workspace, size_t workspace_bytes, void* stream,
                const unsigned long long* tree_masks = nullptr);
}  // namespace

int mla_decode_attend(const int32_t* plan_host, const int32_t* plan_dev, const void* q_nope,
                      const void* q_rope, const void* kv_cache, int64_t num_slots,
                      const int32_t* kv_indptr, const int32_t* kv_indices, float sm_scale, void* out,
                      int32_t out_dtype, float* lse, void* workspace, size_t workspace_bytes,
                      void* stream) {
  return attend_impl(plan_host, plan_dev, 1, q_nope, q_rope, kv_cache, num_slots, kv_indptr, kv_indices, sm_scale,
                     out, out_dtype, lse, workspace, workspace_bytes, stream);
}

int mla_decode_run_multi_query(const int32_t* plan_host, const int32_t* plan_dev, int32_t q_len,
                               const void* q_nope, const void* q_rope, const void* kv_cache, int64_t num_slots,
                               const int32_t* kv_indptr, const int32_t* kv_indices, float sm_scale, void* out,
                               int32_t out_dtype, float* lse, void* workspace, size_t workspace_bytes,
                               void* stream) {
  const int rc = attend_impl(plan_host, plan_dev, q_len, q_nope, q_rope, kv_cache, num_slots, kv_indptr,
                             kv_indices, sm_scale, out, out_dtype, lse, workspace, workspace_bytes, stream);
  if (rc != MLA_OK) return rc;
  return mla_decode_merge(plan_host, plan_dev, out, out_dtype, lse, workspace, workspace_bytes, stream);
}

int mla_decode_run_tree(const int32_t* plan_host, const int32_t* plan_dev, int32_t q_len,
                        const int32_t* tree_parents, uint64_t* tree_masks, const void* q_nope, const void* q_rope,
                        const void* kv_cache, int64_t num_slots, const int32_t* kv_indptr, const int32_t* kv_indices,
                        float sm_scale, void* out, int32_t out_dtype, float* lse, void* workspace,
                        size_t workspace_bytes, void* stream) {
  const int rc0 = check_run_args(plan_host, plan_dev, out_dtype, workspace, workspace_bytes);
  if (rc0 != MLA_OK) return rc0;
  const int B = plan_host[kHBatch], H = plan_host[kHHeads];
  if (q_len < 1 || H % q_len != 0) return MLA_ERR_INVALID_ARG;
  if (q_len > 64) return MLA_ERR_UNSUPPORTED;
  if (q_len == 1)
    return mla_decode_run(plan_host, plan_dev, q_nope, q_rope, kv_cache, num_slots, kv_indptr, kv_indices, sm_scale,
                          out, out_dtype, lse, workspace, workspace_bytes, stream);
  if (!tree_parents || !tree_masks || (reinterpret_cast<uintptr_t>(tree_masks) & 7u) != 0 ||
      (reinterpret_cast<uintptr_t>(tree_parents) & 3u) != 0)
    return MLA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned long long* masks = reinterpret_cast<unsigned long long*>(tree_masks);
  const int rm = launch_tree_masks(tree_parents, B, q_len, masks, static_cast<int*>(workspace), st);
  if (rm != MLA_OK) return rm;
  const int rc = attend_impl(plan_host, plan_dev, q_len, q_nope, q_rope, kv_cache, num_slots, kv_indptr,
                             kv_indices, sm_scale, out, out_dtype, lse, workspace, workspace_bytes, stream, masks);
  if (rc != MLA_OK) return rc;
  return mla_decode_merge(plan_host, plan_dev, out, out_dtype, lse, workspace, workspace_bytes, stream);
}

namespace {
// Tensor maps for the decode kernel of `variant` and its launch (grid = the
// plan's workers); p is complete but for the maps.
int launch_decode(const DecodeParams& p, int variant, const void* q_nope, const void* q_rope, const void* kv_cache,
                  cudaStream_t st) {
  const int H = p.heads;
  CUtensorMap tm_kv, tm_qn, tm_qr;
  const uint64_t qrows = static_cast<uint64_t>(p.batch) * H;
  if (!make_map(&tm_kv, kv_cache, kRow, static_cast<uint64_t>(p.num_slots), 64, 1)) return MLA_ERR_CUDA;
  // the rope as 32-dim halves (64-byte rows): the few-heads kernel's two
  // folded score halves, the pair kernel's two CTAs
  CUtensorMap tm_kr;
  if (!make_map(&tm_kr, kv_cache, kRow, static_cast<uint64_t>(p.num_slots), 32, 1, CU_TENSOR_MAP_SWIZZLE_64B))
    return MLA_ERR_CUDA;
  if (variant == kVariantSwab) {
    if (!make_map(&tm_qr, q_rope, kRope, qrows, 64, static_cast<uint32_t>(H)) ||
        !make_map(&tm_qn, q_nope, kLatent, qrows, 64, static_cast<uint32_t>(H)))
      return MLA_ERR_CUDA;
    return launch_swab(H, tm_kv, tm_kr, tm_qn, tm_qr, p, p.num_workers, st);
  }
  if (!make_map(&tm_qr, q_rope, kRope, qrows, 32, static_cast<uint32_t>(H), CU_TENSOR_MAP_SWIZZLE_64B))
    return MLA_ERR_CUDA;
  return launch_pair(H, tm_kv, tm_kr, tm_qr, p, p.num_workers, st);
}

int attend_impl(const int32_t* plan_host, const int32_t* plan_dev, int32_t q_len, const void* q_nope,
                const void* q_rope, const void* kv_cache, int64_t num_slots, const int32_t* kv_indptr,
                const int32_t* kv_indices, float sm_scale, void* out, int32_t out_dtype, float* lse,
                void* workspace, size_t workspace_bytes, void* stream, const unsigned long long* tree_masks) {
  const int rc0 = check_run_args(plan_host, plan_dev, out_dtype, workspace, workspace_bytes);
  if (rc0 != MLA_OK) return rc0;
  if (!std::isfinite(sm_scale)) return MLA_ERR_INVALID_ARG;
  const int B = plan_host[kHBatch], H = plan_host[kHHeads];
  if (B == 0 || plan_host[kHItems] == 0) return MLA_OK;
  if (!q_nope || !q_rope || !kv_cache || !kv_indptr || !kv_indices || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(kv_cache) || !aligned16(out) ||
      !aligned16(kv_indices) || (lse && !aligned16(lse)))
    return MLA_ERR_INVALID_ARG;
  if (num_slots < 1 || num_slots > 0x7FFFFFFFll) return MLA_ERR_INVALID_ARG;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeParams p{};
  p.plan = plan_dev;
  p.kv_indptr = kv_indptr;
  p.kv_indices = kv_indices;
  p.q_nope = static_cast<const uint16_t*>(q_nope);
  p.kv_cache = static_cast<const uint8_t*>(kv_cache);
  p.out = out;
  p.lse = lse;
  p.part_o = reinterpret_cast<float*>(ws + ws_part_o_offset());
  p.part_lse = reinterpret_cast<float*>(ws + ws_part_lse_offset(plan_host));
  p.status = reinterpret_cast<int*>(ws);
  p.num_slots = num_slots;
  p.batch = B;
  p.heads = H;
  p.out_bf16 = out_dtype;
  p.items_off = plan_items_off(plan_host);
  p.num_workers = plan_host[kHWorkers];
  p.max_partials = plan_host[kHPartials];
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  // multi-query: the plan's head count is q_len x the heads of one query;
  // both decode kernels apply the per-row causal limit
  if (q_len < 1 || H % q_len != 0) return MLA_ERR_INVALID_ARG;
  p.q_len = q_len;
  p.tree_masks = q_len > 1 ? tree_masks : nullptr;   // draft trees: ancestor masks instead of the chain's limit
  return launch_decode(p, plan_host[kHVariant], q_nope, q_rope, kv_cache, st);
}
}  // namespace

int mla_decode_merge(const int32_t* plan_host, const int32_t* plan_dev, void* out, int32_t out_dtype,
                     float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  const int rc0 = check_run_args(plan_host, plan_dev, out_dtype, workspace, workspace_bytes);
  if (rc0 != MLA_OK) return rc0;
  if (plan_host[kHBatch] == 0 || plan_host[kHMerges] == 0) return MLA_OK;
  if (!out || !aligned16(out) || (lse && !aligned16(lse))) return MLA_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  MergeParams m{};
  m.part_o = reinterpret_cast<const float*>(ws + ws_part_o_offset());
  m.part_lse = reinterpret_cast<const float*>(ws + ws_part_lse_offset(plan_host));
  m.list = plan_dev + plan_merge_off(plan_host);
  m.indptr = nullptr;
  m.n_entries = plan_host[kHMerges];
  m.heads = plan_host[kHHeads];
  m.out = out;
  m.out_bf16 = out_dtype;
  m.lse = lse;
  const int32_t* ml = plan_host + plan_merge_off(plan_host);
  int max_pieces = 0;
  for (int i = 0; i < m.n_entries; ++i) max_pieces = std::max(max_pieces, ml[3 * i + 2] - ml[3 * i + 1]);
  return launch_merge(m, m.n_entries, max_pieces, reinterpret_cast<cudaStream_t>(stream));
}

int mla_decode_run(const int32_t* plan_host, const int32_t* plan_dev, const void* q_nope,
                   const void* q_rope, const void* kv_cache, int64_t num_slots,
                   const int32_t* kv_indptr, const int32_t* kv_indices, float sm_scale, void* out,
                   int32_t out_dtype, float* lse, void* workspace, size_t workspace_bytes,
                   void* stream) {
  const int rc = mla_decode_attend(plan_host, plan_dev, q_nope, q_rope, kv_cache, num_slots, kv_indptr,
                                   kv_indices, sm_scale, out, out_dtype, lse, workspace, workspace_bytes,
                                   stream);
  if (rc != MLA_OK) return rc;
  return mla_decode_merge(plan_host, plan_dev, out, out_dtype, lse, workspace, workspace_bytes, stream);
}

namespace {
// Device staging of one host-buffer step: plan words, q_nope, q_rope,
// kv_indptr, kv_indices, out, lse; each region 256-byte aligned.
struct StepLayout {
  size_t plan, qn, qr, ptr, idx, out, lse, total;
};
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
StepLayout step_layout(int32_t B, int32_t H, int64_t nnz, size_t plan_words, int32_t out_dtype) {
  StepLayout l{};
  size_t o = 0;
  l.plan = o; o = align256(o + plan_words * 4);
  l.qn = o;   o = align256(o + static_cast<size_t>(B) * H * kLatent * 2);
  l.qr = o;   o = align256(o + static_cast<size_t>(B) * H * kRope * 2);
  l.ptr = o;  o = align256(o + static_cast<size_t>(B + 1) * 4);
  l.idx = o;  o = align256(o + static_cast<size_t>(nnz) * 4);
  l.out = o;  o = align256(o + static_cast<size_t>(B) * H * kLatent * (out_dtype ? 2 : 4));
  l.lse = o;  o = align256(o + static_cast<size_t>(B) * H * 4);
  l.total = o;
  return l;
}
}  // namespace

size_t mla_step_staging_bytes(int32_t batch, int32_t num_heads, int64_t nnz, size_t plan_words, int32_t out_dtype) {
  if (batch < 0 || num_heads < 1 || nnz < 0) return 0;
  return step_layout(batch, num_heads, nnz, plan_words, out_dtype).total;
}

int mla_decode_step_host(const void* q_nope, const void* q_rope, const int32_t* kv_indptr,
                         const int32_t* kv_indices, int32_t batch, int32_t num_heads, const void* kv_cache,
                         int64_t num_slots, float sm_scale, void* out, int32_t out_dtype, float* lse,
                         int32_t* plan, size_t plan_words, void* staging, size_t staging_bytes, void* workspace,
                         size_t workspace_bytes, void* stream, void* copy_in_stream, void* copy_out_stream) {
  if (!q_nope || !q_rope || !kv_indptr || !out || !lse || !plan || !staging || batch < 1 || out_dtype < 0 ||
      out_dtype > 1)
    return MLA_ERR_INVALID_ARG;
  size_t need = 0, ws_need = 0;
  const int rc = mla_decode_plan(kv_indptr, batch, num_heads, 0, plan, plan_words, &need, &ws_need);
  if (rc != MLA_OK) return rc;
  const int64_t nnz = kv_indptr[batch];
  if (nnz > 0 && !kv_indices) return MLA_ERR_INVALID_ARG;
  const StepLayout l = step_layout(batch, num_heads, nnz, need, out_dtype);
  if (staging_bytes < l.total || workspace_bytes < ws_need) return MLA_ERR_WORKSPACE;
  if (!aligned16(staging)) return MLA_ERR_INVALID_ARG;
  cudaStream_t run_st = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t st = copy_in_stream ? reinterpret_cast<cudaStream_t>(copy_in_stream) : run_st;
  cudaStream_t st_out = copy_out_stream ? reinterpret_cast<cudaStream_t>(copy_out_stream) : run_st;
  // with separate copy streams: the run waits for the copies in, the copies
  // out wait for the run (events from a small per-thread ring, reused round
  // robin; a wait takes the event's state at the time it is issued)
  thread_local cudaEvent_t ring[8] = {};
  thread_local int ring_next = 0;
  cudaEvent_t ev_in = nullptr, ev_run = nullptr;
  for (int i = 0; i < 2; ++i) {
    cudaEvent_t& e = ring[(ring_next + i) % 8];
    if (!e && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return MLA_ERR_CUDA;
  }
  if (st != run_st) ev_in = ring[ring_next];
  if (st_out != run_st) ev_run = ring[(ring_next + 1) % 8];
  ring_next = (ring_next + 2) % 8;
  uint8_t* d = static_cast<uint8_t*>(staging);
  const size_t qn_bytes = static_cast<size_t>(batch) * num_heads * kLatent * 2;
  const size_t qr_bytes = static_cast<size_t>(batch) * num_heads * kRope * 2;
  if (cudaMemcpyAsync(d + l.plan, plan, need * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(d + l.qn, q_nope, qn_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(d + l.qr, q_rope, qr_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(d + l.ptr, kv_indptr, static_cast<size_t>(batch + 1) * 4, cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      (nnz > 0 && cudaMemcpyAsync(d + l.idx, kv_indices, static_cast<size_t>(nnz) * 4, cudaMemcpyHostToDevice, st) !=
                      cudaSuccess)) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (ev_in && (cudaEventRecord(ev_in, st) != cudaSuccess || cudaStreamWaitEvent(run_st, ev_in, 0) != cudaSuccess)) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  const int rr = mla_decode_run(plan, reinterpret_cast<const int32_t*>(d + l.plan), d + l.qn, d + l.qr, kv_cache,
                                num_slots, reinterpret_cast<const int32_t*>(d + l.ptr),
                                reinterpret_cast<const int32_t*>(d + l.idx), sm_scale, d + l.out, out_dtype,
                                reinterpret_cast<float*>(d + l.lse), workspace, workspace_bytes, stream);
  if (rr != MLA_OK) return rr;
  if (ev_run && (cudaEventRecord(ev_run, run_st) != cudaSuccess || cudaStreamWaitEvent(st_out, ev_run, 0) != cudaSuccess)) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  const size_t out_bytes = static_cast<size_t>(batch) * num_heads * kLatent * (out_dtype ? 2 : 4);
  if (cudaMemcpyAsync(out, d + l.out, out_bytes, cudaMemcpyDeviceToHost, st_out) != cudaSuccess ||
      cudaMemcpyAsync(lse, d + l.lse, static_cast<size_t>(batch) * num_heads * 4, cudaMemcpyDeviceToHost, st_out) !=
          cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

int mla_merge_states(const float* v_partial, const float* s_partial, const int32_t* merge_indptr,
                     int32_t batch, int32_t num_heads, void* out, int32_t out_dtype, float* lse,
                     void* stream) {
  if (batch < 0 || num_heads < 1 || num_heads > 65535) return MLA_ERR_INVALID_ARG;
  if (out_dtype != 0 && out_dtype != 1) return MLA_ERR_UNSUPPORTED;
  if (batch == 0) return MLA_OK;
  if (!v_partial || !s_partial || !merge_indptr || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(v_partial) || !aligned16(out) || (lse && !aligned16(lse))) return MLA_ERR_INVALID_ARG;
  MergeParams m{};
  m.part_o = v_partial;
  m.part_lse = s_partial;
  m.list = nullptr;
  m.indptr = merge_indptr;
  m.n_entries = batch;
  m.heads = num_heads;
  m.out = out;
  m.out_bf16 = out_dtype;
  m.lse = lse;
  return launch_merge(m, batch, 0, reinterpret_cast<cudaStream_t>(stream));
}

int mla_absorb_query(const void* q_pre, const void* w_kc, void* q_nope, int32_t batch, int32_t num_heads,
                     int32_t nope_dim, void* workspace, void* stream) {
  if (nope_dim != 128) return MLA_ERR_UNSUPPORTED;
  if (batch < 0 || num_heads < 1 || num_heads > 65535) return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!q_pre || !w_kc || !q_nope || !aligned16(q_pre) || !aligned16(w_kc) || !aligned16(q_nope) ||
      (workspace && !aligned16(workspace)))
    return MLA_ERR_INVALID_ARG;
  const uint64_t H = static_cast<uint64_t>(num_heads);
  CUtensorMap tm_a, tm_w;
  if (!make_map(&tm_a, q_pre, H * 128, static_cast<uint64_t>(batch), 64, 128) ||
      !make_map(&tm_w, w_kc, kLatent, H * 128, 64, 64))
    return MLA_ERR_CUDA;
  HeadGemmParams p{};
  p.out = q_nope;
  p.status = static_cast<int*>(workspace);
  p.rows = batch;
  p.heads = num_heads;
  return launch_absorb(tm_a, tm_w, p, reinterpret_cast<cudaStream_t>(stream));
}

int mla_project_output(const void* o_lat, const void* w_vc, void* out, int32_t out_dtype, int32_t batch,
                       int32_t num_heads, int32_t v_dim, void* workspace, void* stream) {
  if (v_dim != 128 || (out_dtype != 0 && out_dtype != 1)) return MLA_ERR_UNSUPPORTED;
  if (batch < 0 || num_heads < 1 || num_heads > 65535) return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!o_lat || !w_vc || !out || !aligned16(o_lat) || !aligned16(w_vc) || !aligned16(out) ||
      (workspace && !aligned16(workspace)))
    return MLA_ERR_INVALID_ARG;
  const uint64_t H = static_cast<uint64_t>(num_heads);
  CUtensorMap tm_a, tm_w;
  if (!make_map(&tm_a, o_lat, H * kLatent, static_cast<uint64_t>(batch), 64, 128) ||
      !make_map(&tm_w, w_vc, 128, H * kLatent, 64, 64))
    return MLA_ERR_CUDA;
  HeadGemmParams p{};
  p.out = out;
  p.status = static_cast<int*>(workspace);
  p.rows = batch;
  p.heads = num_heads;
  return launch_project(tm_a, tm_w, p, out_dtype, reinterpret_cast<cudaStream_t>(stream));
}

int mla_merge_two_states(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b, int64_t rows,
                         void* out, int32_t out_dtype, float* lse, void* stream) {
  if (out_dtype != 0 && out_dtype != 1) return MLA_ERR_UNSUPPORTED;
  if (rows < 0 || rows > 0x7FFFFFFFll) return MLA_ERR_INVALID_ARG;
  if (rows == 0) return MLA_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !out || !aligned16(o_a) || !aligned16(o_b) || !aligned16(out))
    return MLA_ERR_INVALID_ARG;
  return launch_merge_two(o_a, lse_a, o_b, lse_b, out, out_dtype, lse, rows, reinterpret_cast<cudaStream_t>(stream));
}

int mla_append_kv(void* kv_cache, int64_t num_slots, const int32_t* slots, const void* rows, int32_t batch,
                  void* workspace, void* stream) {
  if (batch < 0 || num_slots < 1) return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!kv_cache || !slots || !rows || !aligned16(kv_cache) || !aligned16(rows) || (workspace && !aligned16(workspace)))
    return MLA_ERR_INVALID_ARG;
  AppendParams p{};
  p.kv_cache = kv_cache;
  p.src = rows;
  p.slots = slots;
  p.status = static_cast<int*>(workspace);
  p.num_slots = num_slots;
  p.rows = batch;
  return launch_append(p, reinterpret_cast<cudaStream_t>(stream));
}

namespace {
// Capacities of a decode whose plan is written into device buffers before
// each CUDA-graph replay: at most max_batch requests on W workers give at
// most max_batch + W - 1 pieces (a request is cut only where a worker is
// full), so at most that many partial states and items and max_batch merge
// entries.
struct GraphSizes {
  int variant, W;
  long long P, words;
  size_t ws, lse_off;
};
int graph_sizes(int32_t max_batch, int32_t H, int32_t num_sms, GraphSizes* g) {
  int T = 0, cpw = 0;
  if (max_batch < 1 || num_sms < 1) return MLA_ERR_INVALID_ARG;
  g->variant = variant_for_heads(H, &T, &cpw);
  if (!g->variant) return MLA_ERR_UNSUPPORTED;
  g->W = num_sms / cpw;
  if (g->W < 1) return MLA_ERR_INVALID_ARG;
  g->P = static_cast<long long>(max_batch) + g->W - 1;
  g->words = kHeaderWords + (g->W + 1ll) + 4ll * g->P + 3ll * max_batch;
  g->lse_off = kWsHeaderBytes + static_cast<size_t>(g->P) * H * kLatent * 4;
  g->ws = (g->lse_off + static_cast<size_t>(g->P) * H * 4 + 255) / 256 * 256;
  if (g->words > (1ll << 31) - 1) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}
}  // namespace

int mla_decode_graph_sizes(int32_t max_batch, int32_t num_heads, int32_t num_sms, size_t* plan_words,
                           size_t* workspace_bytes) {
  GraphSizes g{};
  const int rc = graph_sizes(max_batch, num_heads, num_sms, &g);
  if (rc != MLA_OK) return rc;
  if (plan_words) *plan_words = static_cast<size_t>(g.words);
  if (workspace_bytes) *workspace_bytes = g.ws;
  return MLA_OK;
}

int mla_decode_run_graph(const int32_t* plan_dev, size_t plan_words, int32_t max_batch, int32_t num_heads,
                         int32_t num_sms, const void* q_nope, const void* q_rope, const void* kv_cache,
                         int64_t num_slots, const int32_t* kv_indptr, const int32_t* kv_indices, float sm_scale,
                         void* out, int32_t out_dtype, float* lse, void* workspace, size_t workspace_bytes,
                         void* stream) {
  GraphSizes g{};
  const int rc0 = graph_sizes(max_batch, num_heads, num_sms, &g);
  if (rc0 != MLA_OK) return rc0;
  if (out_dtype != 0 && out_dtype != 1) return MLA_ERR_UNSUPPORTED;
  if (!plan_dev || !q_nope || !q_rope || !kv_cache || !kv_indptr || !kv_indices || !out || !workspace)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(kv_cache) || !aligned16(out) || !aligned16(kv_indices) ||
      !aligned16(workspace) || (lse && !aligned16(lse)))
    return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale) || num_slots < 1 || num_slots > 0x7FFFFFFFll) return MLA_ERR_INVALID_ARG;
  if (plan_words < static_cast<size_t>(g.words) || workspace_bytes < g.ws) return MLA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeParams p{};
  p.plan = plan_dev;
  p.kv_indptr = kv_indptr;
  p.kv_indices = kv_indices;
  p.q_nope = static_cast<const uint16_t*>(q_nope);
  p.kv_cache = static_cast<const uint8_t*>(kv_cache);
  p.out = out;
  p.lse = lse;
  p.part_o = reinterpret_cast<float*>(ws + kWsHeaderBytes);
  p.part_lse = reinterpret_cast<float*>(ws + g.lse_off);
  p.status = reinterpret_cast<int*>(ws);
  p.num_slots = num_slots;
  p.batch = max_batch;
  p.heads = num_heads;
  p.out_bf16 = out_dtype;
  p.items_off = kHeaderWords + g.W + 1;
  p.num_workers = g.W;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.q_len = 1;
  p.plan_cap_words = static_cast<int>(g.words);
  p.max_partials = static_cast<int>(g.P);
  const int rc = launch_decode(p, g.variant, q_nope, q_rope, kv_cache, st);
  if (rc != MLA_OK) return rc;
  MergeParams m{};
  m.part_o = p.part_o;
  m.part_lse = p.part_lse;
  m.list = nullptr;
  m.indptr = nullptr;
  m.n_entries = max_batch;
  m.heads = num_heads;
  m.out = out;
  m.out_bf16 = out_dtype;
  m.lse = lse;
  m.plan = plan_dev;
  m.plan_cap_words = static_cast<int>(g.words);
  m.batch = max_batch;
  m.max_partials = static_cast<int>(g.P);
  m.workers = g.W;
  m.status = p.status;
  return launch_merge(m, max_batch, 16, st);
}

namespace {
// FP8 decode workspace: the plan's workspace, then the query images [B] and
// the per-head factors [B, H], each 256-byte aligned.
struct Fp8WsLayout {
  size_t img, fac, total;
};
Fp8WsLayout fp8_ws_layout(const int32_t* plan_host) {
  Fp8WsLayout l{};
  const size_t B = static_cast<size_t>(plan_host[kHBatch]), H = static_cast<size_t>(plan_host[kHHeads]);
  l.img = (ws_needed_bytes(plan_host) + 255) & ~size_t(255);
  l.fac = (l.img + B * fp8_image_bytes(static_cast<int>(H)) + 255) & ~size_t(255);
  l.total = l.fac + B * H * 4;
  return l;
}
}  // namespace

int mla_decode_fp8_workspace_bytes(const int32_t* plan_host, size_t* workspace_bytes) {
  if (!plan_header_ok(plan_host) || !workspace_bytes) return MLA_ERR_INVALID_ARG;
  *workspace_bytes = fp8_ws_layout(plan_host).total;
  return MLA_OK;
}

int mla_decode_run_fp8(const int32_t* plan_host, const int32_t* plan_dev, const void* q_nope, const void* q_rope,
                       const void* kv_cache, int64_t num_slots, float kv_scale, const int32_t* kv_indptr,
                       const int32_t* kv_indices, float sm_scale, void* out, int32_t out_dtype, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan_header_ok(plan_host) || !plan_dev) return MLA_ERR_INVALID_ARG;
  if (out_dtype != 0 && out_dtype != 1) return MLA_ERR_UNSUPPORTED;
  if (!std::isfinite(sm_scale) || !std::isfinite(kv_scale) || !(kv_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  const Fp8WsLayout wl = fp8_ws_layout(plan_host);
  if (!workspace || !aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < wl.total) return MLA_ERR_WORKSPACE;
  const int B = plan_host[kHBatch], H = plan_host[kHHeads];
  if (B == 0 || plan_host[kHItems] == 0)
    return mla_decode_merge(plan_host, plan_dev, out, out_dtype, lse, workspace, workspace_bytes, stream);
  if (!q_nope || !q_rope || !kv_cache || !kv_indptr || !kv_indices || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(kv_cache) || !aligned16(out) ||
      !aligned16(kv_indices) || (lse && !aligned16(lse)))
    return MLA_ERR_INVALID_ARG;
  if (num_slots < 1 || num_slots > 0x7FFFFFFFll) return MLA_ERR_INVALID_ARG;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeParams p{};
  p.plan = plan_dev;
  p.kv_indptr = kv_indptr;
  p.kv_indices = kv_indices;
  p.q_nope = static_cast<const uint16_t*>(q_nope);
  p.q_rope = static_cast<const uint16_t*>(q_rope);
  p.kv_cache = static_cast<const uint8_t*>(kv_cache);
  p.out = out;
  p.lse = lse;
  p.part_o = reinterpret_cast<float*>(ws + ws_part_o_offset());
  p.part_lse = reinterpret_cast<float*>(ws + ws_part_lse_offset(plan_host));
  p.status = reinterpret_cast<int*>(ws);
  p.num_slots = num_slots;
  p.batch = B;
  p.heads = H;
  p.out_bf16 = out_dtype;
  p.items_off = plan_items_off(plan_host);
  p.num_workers = plan_host[kHWorkers];
  p.max_partials = plan_host[kHPartials];
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.q_len = 1;
  Fp8Params p8{};
  p8.img = ws + wl.img;
  p8.fac = reinterpret_cast<const float*>(ws + wl.fac);
  p8.kv_scale = kv_scale;
  Fp8PrepParams pp{};
  pp.q_nope = static_cast<const uint16_t*>(q_nope);
  pp.q_rope = static_cast<const uint16_t*>(q_rope);
  pp.img = ws + wl.img;
  pp.fac = reinterpret_cast<float*>(ws + wl.fac);
  pp.rows = B * H;
  // 8-bit maps over the cache: 128-byte latent boxes and 32-byte rope boxes
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MLA_ERR_CUDA;
  CUtensorMap tm_lat, tm_rope;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRow), static_cast<cuuint64_t>(num_slots)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRow)};
  cuuint32_t box_lat[2] = {128, 1}, box_rope[2] = {32, 1}, estr[2] = {1, 1};
  if (fn(&tm_lat, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv_cache), dims, strides, box_lat, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      fn(&tm_rope, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv_cache), dims, strides, box_rope, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MLA_ERR_CUDA;
  const int rc = plan_host[kHVariant] == kVariantSwab ? launch_swab8(H, tm_lat, tm_rope, p, p8, pp, plan_host[kHWorkers], st)
                                                        : launch_pair8(H, tm_lat, tm_rope, p, kv_scale,
                                                                       plan_host[kHWorkers], st);
  if (rc != MLA_OK) return rc;
  return mla_decode_merge(plan_host, plan_dev, out, out_dtype, lse, workspace, workspace_bytes, stream);
}

int mla_append_kv_fp8(void* kv_cache, int64_t num_slots, const int32_t* slots, const void* rows, int32_t batch,
                      float kv_scale, void* workspace, void* stream) {
  if (batch < 0 || num_slots < 1 || !std::isfinite(kv_scale) || !(kv_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!kv_cache || !slots || !rows || !aligned16(kv_cache) || !aligned16(rows) || (workspace && !aligned16(workspace)))
    return MLA_ERR_INVALID_ARG;
  AppendFp8Params p{};
  p.kv_cache = static_cast<uint8_t*>(kv_cache);
  p.src = static_cast<const uint16_t*>(rows);
  p.slots = slots;
  p.status = static_cast<int*>(workspace);
  p.num_slots = num_slots;
  p.rows = batch;
  p.kv_scale = kv_scale;
  return launch_append_fp8(p, reinterpret_cast<cudaStream_t>(stream));
}

int mla_check_errors(void* workspace, void* stream) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  int status = 0;
  if (cudaMemcpy(&status, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (status != 0) {
    if (cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
  }
  return status;
}

}  // extern "C"
