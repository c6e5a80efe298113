// Ancestor masks of draft trees for tree-shaped verification ("[sglang] EAGLE
// 트리 검증 어텐션 최적화", section "들어가며": each query token attends to its
// own ancestor chain among the drafts).  One thread per draft: walk the
// parent links from the draft to the root, setting the bit of every draft on
// the way (the draft's own bit included).  A parent must be an earlier
// draft, so each step moves to a smaller index and the walk ends within W
// steps; a link that does not is recorded as MLA_ERR_TREE and the draft keeps
// only its own bit (a child of the context).
#include "mla_device.cuh"
#include "mla_launch.h"

namespace mla {
namespace {

__global__ void __launch_bounds__(64) tree_mask_kernel(const int32_t* __restrict__ parents, int batch, int width,
                                                      unsigned long long* __restrict__ masks, int* status) {
  const int b = blockIdx.x, i = threadIdx.x;
  if (b >= batch || i >= width) return;
  const int32_t* par = parents + static_cast<size_t>(b) * width;
  unsigned long long m = 1ull << i;
  int x = i;
  for (int step = 0; step < width; ++step) {
    const int px = __ldg(par + x);
    if (px < 0) {
      if (px != -1) { m = 1ull << i; record_status(status, MLA_ERR_TREE); }
      break;
    }
    if (px >= x) {                                // not an earlier draft
      m = 1ull << i;
      record_status(status, MLA_ERR_TREE);
      break;
    }
    m |= 1ull << px;
    x = px;
  }
  masks[static_cast<size_t>(b) * width + i] = m;
}

}  // namespace

int launch_tree_masks(const int32_t* parents, int batch, int width, unsigned long long* masks, int* status,
                      cudaStream_t stream) {
  if (batch <= 0) return MLA_OK;
  if (width < 1 || width > 64) return MLA_ERR_UNSUPPORTED;
  tree_mask_kernel<<<batch, 64, 0, stream>>>(parents, batch, width, masks, status);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace mla
