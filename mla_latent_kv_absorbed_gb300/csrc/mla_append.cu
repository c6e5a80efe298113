// Cache append of a decode step: request b's new 576-wide row (latent, then
// rope key) goes to cache slot slots[b] ("实现差距：MLA 与 DeepSeek V3",
// section 2.4: the Pallas V2 kernel writes the new token's kv_c and k_pe into
// the cache before attending).  The row is 1152 bytes = 72 16-byte pieces:
// one thread per piece, four rows per 288-thread block, so a warp stores 512
// contiguous bytes.  A slot outside [0, num_slots) is skipped and recorded as
// MLA_ERR_INDEX_OOB in the status word when one is given.
#include "mla_device.cuh"
#include "mla_launch.h"

namespace mla {

constexpr int kAppendPieces = kRow * 2 / 16;     // 72
constexpr int kAppendRows = 4;

__global__ void __launch_bounds__(kAppendPieces * kAppendRows) append_kernel(const AppendParams p) {
  const int r = blockIdx.x * kAppendRows + threadIdx.x / kAppendPieces;
  const int piece = threadIdx.x % kAppendPieces;
  // a programmatic dependent of the previous kernel in the stream: read and
  // write only once it has finished, and let the next one be scheduled
  griddep_wait();
  griddep_launch_dependents();
  if (r >= p.rows) return;
  const long long slot = __ldg(p.slots + r);
  if (slot < 0 || slot >= p.num_slots) {
    if (piece == 0) record_status(p.status, MLA_ERR_INDEX_OOB);
    return;
  }
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.src) + static_cast<size_t>(r) * kAppendPieces + piece);
  reinterpret_cast<uint4*>(p.kv_cache)[slot * kAppendPieces + piece] = v;
}

int launch_append(const AppendParams& p, cudaStream_t stream) {
  if (p.rows <= 0) return MLA_OK;
  const int blocks = (p.rows + kAppendRows - 1) / kAppendRows;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(kAppendPieces * kAppendRows, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, append_kernel, p) != cudaSuccess) return MLA_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace mla
