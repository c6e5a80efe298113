// Flash-Decoding merge of split-KV partial states by LSE rescaling
// ("Attention backends", paragraph "FlashAttention": keys split across
// blocks, partial results merged with the same rescaling).
//
// For one request and head with partial states (o_i, lse_i), each o_i already
// divided by its own softmax sum:
//   M = max_i lse_i,  w_i = exp(lse_i - M),
//   out = sum_i w_i o_i / sum_i w_i,  lse = M + ln sum_i w_i.
// Partials with lse_i = -inf weigh nothing; no live partial gives out = 0,
// lse = -inf (an empty request).
//
// One 128-thread block per (entry, head); each thread owns four latent dims
// and reads them as one float4 per partial, so the partials stream through
// in coalesced 2 KB rows.
#include <cuda_bf16.h>

#include "mla_launch.h"

namespace mla {

__global__ void __launch_bounds__(128) merge_kernel(const MergeParams p) {
  const int e = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  int b, p0, p1;
  if (p.list) {
    b = p.list[3 * e];
    p0 = p.list[3 * e + 1];
    p1 = p.list[3 * e + 2];
  } else {
    b = e;
    p0 = p.indptr[e];
    p1 = p.indptr[e + 1];
  }
  const int H = p.heads;
  float M = -INFINITY;
  for (int i = p0; i < p1; ++i) M = fmaxf(M, __ldg(p.part_lse + static_cast<size_t>(i) * H + h));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (M > -INFINITY) {
    for (int i = p0; i < p1; ++i) {
      const float l = __ldg(p.part_lse + static_cast<size_t>(i) * H + h);
      const float w = (l == -INFINITY) ? 0.f : expf(l - M);
      const float4 v = __ldg(reinterpret_cast<const float4*>(
                                 p.part_o + (static_cast<size_t>(i) * H + h) * kLatent) + tid);
      wsum += w;
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const size_t o = (static_cast<size_t>(b) * H + h) * kLatent + 4 * tid;
  if (p.out_bf16) {
    __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(p.out) + o);
    dst[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    dst[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  if (tid == 0 && p.lse) p.lse[static_cast<size_t>(b) * H + h] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

int launch_merge(const MergeParams& p, int entries, cudaStream_t stream) {
  if (entries <= 0) return MLA_OK;
  dim3 grid(entries, p.heads);
  merge_kernel<<<grid, 128, 0, stream>>>(p);
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace mla
