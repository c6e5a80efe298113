// The failure path of the kernels' bounded waits, on its own.  Every decode
// and head-product kernel waits on its mbarriers through mbar_wait,
// which gives up after MLA_WAIT_LIMIT_NS of wall time, records
// MLA_ERR_TIMEOUT in the workspace status word and lets the kernel return, so
// a stalled pipeline ends as a status code instead of a hung GPU.  In those
// kernels every wait completes in normal use; this kernel waits on a barrier
// that nothing ever completes, so that a test can see the limit end the wait,
// the status reach the host and the context stay usable.  It touches nothing
// but its own shared memory and the status word.
#include "mla_device.cuh"

namespace mla {
namespace {

__global__ void __launch_bounds__(32, 1) probe_wait_limit_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar_word;
  __shared__ int abort_flag;
  const uint32_t bar = smem_u32(&bar_word);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);         // one arrival expected; none is ever made
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    const WaitCtx wc{&abort_flag, status};
    mbar_wait(bar, 0, wc);     // phase 0 never completes: returns false after the limit
  }
}

}  // namespace
}  // namespace mla

extern "C" int mla_probe_wait_limit(void* workspace, void* stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return MLA_ERR_INVALID_ARG;
  mla::probe_wait_limit_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<int*>(workspace));
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
