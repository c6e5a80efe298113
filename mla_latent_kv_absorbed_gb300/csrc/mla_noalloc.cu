// mla_decode_run_noalloc: the decode step for callers that cannot allocate
// device memory.  The split-KV partial states and the device status word live
// in one static device buffer of the library image instead of a caller
// workspace (see include/mla_decode.h for the contract).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "mla_internal.h"
#include "mla_plan.h"

namespace {

constexpr size_t kScratchBytes = MLA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

}  // namespace

// One buffer per device that loads the library; held until process exit.
// Static initialisation leaves it zero, so its status word starts clear.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry point (the library does
// not link the driver API directly).
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the buffer on the current device, looked up with that
// device current.  Host code must not use the symbol itself: on the host it
// names a stand-in, not device memory.  The address belongs to the module
// loaded in the device's current context, so the cache is keyed on that
// context as well: after cudaDeviceReset (or anything else that replaces the
// primary context and reloads the module) the next call looks it up again.
void* scratch_on_current_device() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  static CUcontext ctx_of[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  const CtxGetCurrentFn get = ctx_get_current_fn();
  if (!get) return nullptr;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return nullptr;   // null before the device's first runtime call
  std::lock_guard<std::mutex> lock(mu);
  if (!ctx || !addr[dev] || ctx_of[dev] != ctx) {
    // the symbol query makes the device's primary context current if it is
    // not yet, so the context read after it is the one the address lives in
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      addr[dev] = nullptr;
      return nullptr;
    }
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
    addr[dev] = p;
    ctx_of[dev] = ctx;
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
  // The status word is not cleared here: like a caller workspace's, it keeps
  // the first device-side error until mla_noalloc_check_errors reads it.
  return mla_decode_run(plan_host, plan_dev, q_nope, q_rope, kv_cache, num_slots, kv_indptr, kv_indices, sm_scale,
                        out, out_dtype, lse, ws, kScratchBytes, stream);
}

extern "C" int mla_noalloc_check_errors(void* stream) {
  void* ws = scratch_on_current_device();
  if (!ws) return MLA_ERR_CUDA;
  // reads and clears the static buffer's status word, as mla_check_errors
  // does for a caller workspace (a synchronising copy into a host int: no
  // allocation)
  return mla_check_errors(ws, stream);
}
