// mla_decode_run_noalloc: the decode step for callers that cannot allocate
// device memory.  The split-KV partial states and the device status word live
// in one static device buffer of the library image instead of a caller
// workspace (see include/mla_decode.h for the contract).
#include <cuda_runtime.h>

#include <mutex>

#include "mla_internal.h"
#include "mla_plan.h"

namespace {

constexpr size_t kScratchBytes = MLA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

}  // namespace

// One buffer per device that loads the library; held until process exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

// Device address of the buffer on the current device, looked up once per
// device with that device current.  Host code must not use the symbol itself:
// on the host it names a stand-in, not device memory.
void* scratch_on_current_device() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int mla_decode_run_noalloc(const int32_t* plan_host, const int32_t* plan_dev, const void* q_nope,
                                      const void* q_rope, const void* kv_cache, int64_t num_slots,
                                      const int32_t* kv_indptr, const int32_t* kv_indices, float sm_scale,
                                      void* out, int32_t out_dtype, float* lse, void* stream) {
  using namespace mla;
  if (!plan_host || plan_host[kHMagic] != kPlanMagic) return MLA_ERR_INVALID_ARG;
  if (plan_host[kHPartials] < 0 || plan_host[kHHeads] < 1 || plan_host[kHBatch] < 0) return MLA_ERR_INVALID_ARG;
  const size_t need = ws_needed_bytes(plan_host);
  if (need > kScratchBytes) return MLA_ERR_WORKSPACE;
  void* ws = scratch_on_current_device();
  if (!ws) return MLA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, kWsHeaderBytes, st) != cudaSuccess) {   // the status word starts at zero
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return mla_decode_run(plan_host, plan_dev, q_nope, q_rope, kv_cache, num_slots, kv_indptr, kv_indices, sm_scale,
                        out, out_dtype, lse, ws, kScratchBytes, stream);
}
