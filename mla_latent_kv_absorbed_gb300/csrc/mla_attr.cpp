// Per-device launch settings shared by the kernel launchers: the dynamic
// shared-memory limit of each kernel and the SM count.  Both are looked up
// once and reused; a process may drive several devices from several host
// threads, so the caches are keyed on the context (the limit) or the device
// (the SM count) and safe to use concurrently.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "mla_launch.h"

namespace mla {
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

CUcontext current_context() {
  CUcontext ctx = nullptr;
  const CtxGetCurrentFn get = ctx_get_current_fn();
  if (!get || get(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

}  // namespace

bool set_smem_limit(const void* func, int bytes) {
  // The attribute belongs to the function as loaded in one context: remember
  // the (function, context) pairs it was set in.  A context made after a
  // device reset is a new one and gets the attribute again.
  static std::mutex mu;
  static std::vector<std::pair<const void*, CUcontext>> done;
  CUcontext ctx = current_context();   // null before the device's first runtime call: set it then
  if (ctx) {
    std::lock_guard<std::mutex> lock(mu);
    for (const auto& e : done)
      if (e.first == func && e.second == ctx) return true;
  }
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  ctx = current_context();             // the call above made a context current if none was
  if (ctx) {
    std::lock_guard<std::mutex> lock(mu);
    done.emplace_back(func, ctx);
  }
  return true;
}

int device_sm_count() {
  // queried once per device ordinal; a race only repeats the query
  static std::atomic<int> sms_of[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int cached = (dev >= 0 && dev < 64) ? sms_of[dev].load(std::memory_order_relaxed) : 0;
  if (cached > 0) return cached;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return 0;
  }
  if (dev >= 0 && dev < 64) sms_of[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace mla
