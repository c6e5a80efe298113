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
// One block per (entry, head) of G groups of 128 threads (G = 1, 2 or 4, from
// the most pieces an entry has).  The partial LSEs are loaded in parallel and
// their weights go through shared memory; then thread t of group k owns latent
// dims 4t..4t+3 and streams the partials k, k+G, k+2G, ... as float4, four at a
// time, so 4G partial rows per dim are in flight and a request cut into tens of
// pieces costs a few memory round trips.  The groups' sums are added in a
// fixed order.
// The kernel is launched as a programmatic dependent of the decode kernel:
// its blocks are scheduled while the decode kernel drains and wait
// (griddepcontrol.wait) until its partial states are complete and visible.
#include <cuda_bf16.h>

#include "mla_device.cuh"
#include "mla_launch.h"

namespace mla {

constexpr int kMergeGroups = 4;                      // at most
constexpr int kMergeThreads = 128 * kMergeGroups;
constexpr int kMergeChunk = 1024;   // partials whose weights one pass keeps in shared memory

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
  __shared__ float s_w[kMergeChunk];
  __shared__ float s_red[kMergeThreads / 32];
  __shared__ float4 s_acc[kMergeGroups - 1][128];
  __shared__ float s_wsum[kMergeGroups - 1];
  const int e = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int G = static_cast<int>(blockDim.x >> 7), grp = tid >> 7, t = tid & 127;
  // the next kernel in the stream may be scheduled now; it waits for this
  // grid before it touches what this grid reads or writes
  griddep_launch_dependents();
  const int nthreads = static_cast<int>(blockDim.x);
  int b, p0, p1;
  if (p.plan) {
    // device-only plan (graph replays): the entry count, the list and its
    // bounds come from the plan words; the grid covers every possible entry
    const int32_t* h = p.plan;
    const int W = h[kHWorkers], n_items = h[kHItems], n_merges = h[kHMerges];
    const long long off = kHeaderWords + static_cast<long long>(W) + 1 + 4ll * n_items;
    const bool good = h[kHMagic] == kPlanMagic && h[kHVersion] == kPlanVersion && h[kHHeads] == p.heads &&
                      W == p.workers &&
                      n_items >= 0 && n_merges >= 0 && off + 3ll * n_merges <= p.plan_cap_words;
    if (!good || e >= n_merges) return;
    b = h[off + 3 * e];
    p0 = h[off + 3 * e + 1];
    p1 = h[off + 3 * e + 2];
    if (b < 0 || b >= p.batch || p0 < 0 || p1 < p0 || p1 > p.max_partials) {
      if (tid == 0) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
      return;
    }
  } else if (p.list) {
    b = p.list[3 * e];
    p0 = p.list[3 * e + 1];
    p1 = p.list[3 * e + 2];
  } else {
    b = e;
    p0 = p.indptr[e];
    p1 = p.indptr[e + 1];
  }
  griddep_wait();
  const int H = p.heads;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f, M = -INFINITY;
  for (int c0 = p0; c0 < p1; c0 += kMergeChunk) {
    // this chunk's partials: LSEs in parallel, then the chunk maximum
    const int nc = min(kMergeChunk, p1 - c0);
    float m = -INFINITY;
    for (int i = tid; i < nc; i += nthreads) {
      const float l = __ldcg(p.part_lse + static_cast<size_t>(c0 + i) * H + h);
      s_w[i] = l;
      m = fmaxf(m, l);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((tid & 31) == 0) s_red[tid >> 5] = m;
    __syncthreads();
    float mc = s_red[0];
    for (int w = 1; w < nthreads / 32; ++w) mc = fmaxf(mc, s_red[w]);
    // fold the chunk into the running state (one chunk unless a request has
    // more than kMergeChunk partials)
    const float mn = fmaxf(M, mc);
    if (mn > -INFINITY && M > -INFINITY && mn != M) {
      const float a = expf(M - mn);
      wsum *= a;
      acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
    }
    M = mn;
    for (int i = tid; i < nc; i += nthreads) {
      const float l = s_w[i];
      s_w[i] = (l == -INFINITY || M == -INFINITY) ? 0.f : expf(l - M);
    }
    __syncthreads();
    const float4* src = reinterpret_cast<const float4*>(p.part_o + (static_cast<size_t>(c0) * H + h) * kLatent) + t;
    const size_t stride = static_cast<size_t>(H) * kLatent / 4;   // float4 per partial
    int i = grp;
    for (; i + 3 * G < nc; i += 4 * G) {
      float4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = __ldcg(src + (i + q * G) * stride);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float w = s_w[i + q * G];
        wsum += w;
        acc.x = fmaf(w, v[q].x, acc.x);
        acc.y = fmaf(w, v[q].y, acc.y);
        acc.z = fmaf(w, v[q].z, acc.z);
        acc.w = fmaf(w, v[q].w, acc.w);
      }
    }
    for (; i < nc; i += G) {
      const float4 v = __ldcg(src + i * stride);
      const float w = s_w[i];
      wsum += w;
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    __syncthreads();   // s_w and s_red are reused by the next chunk
  }
  // add the groups' sums in a fixed order
  if (grp > 0) {
    s_acc[grp - 1][t] = acc;
    if (t == 0) s_wsum[grp - 1] = wsum;
  }
  __syncthreads();
  if (grp != 0) return;
  for (int k = 0; k < G - 1; ++k) {
    const float4 a = s_acc[k][t];
    acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
    wsum += s_wsum[k];
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const size_t o = (static_cast<size_t>(b) * H + h) * kLatent + 4 * t;
  if (p.out_bf16) {
    __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(p.out) + o);
    dst[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    dst[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  if (t == 0 && p.lse) p.lse[static_cast<size_t>(b) * H + h] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

// Two states per row, same layout ([rows, 512] and [rows]): the merge of a
// shared-prefix pass with a per-request suffix pass (the EAGLE tree-verify
// page's prefix / suffix attention merged by LSE).  One 128-thread block per
// row, four dims per thread; out may be the first state's array.
__global__ void __launch_bounds__(128) merge_two_kernel(const float* __restrict__ o_a, const float* __restrict__ l_a,
                                                        const float* __restrict__ o_b, const float* __restrict__ l_b,
                                                        void* out, int out_bf16, float* lse, long long rows) {
  const long long r = blockIdx.x;
  if (r >= rows) return;
  const float la = __ldg(l_a + r), lb = __ldg(l_b + r);
  const float m = fmaxf(la, lb);
  const float wa = la == -INFINITY ? 0.f : expf(la - m), wb = lb == -INFINITY ? 0.f : expf(lb - m);
  const float ws = wa + wb, inv = ws > 0.f ? 1.f / ws : 0.f;
  const float4 a = reinterpret_cast<const float4*>(o_a + r * kLatent)[threadIdx.x];
  const float4 b = reinterpret_cast<const float4*>(o_b + r * kLatent)[threadIdx.x];
  const float4 v = make_float4((wa * a.x + wb * b.x) * inv, (wa * a.y + wb * b.y) * inv, (wa * a.z + wb * b.z) * inv,
                               (wa * a.w + wb * b.w) * inv);
  if (out_bf16) {
    __nv_bfloat162* d = reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(out) + r * kLatent) +
                        2 * threadIdx.x;
    d[0] = __floats2bfloat162_rn(v.x, v.y);
    d[1] = __floats2bfloat162_rn(v.z, v.w);
  } else {
    reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + r * kLatent)[threadIdx.x] = v;
  }
  if (threadIdx.x == 0 && lse) lse[r] = ws > 0.f ? m + logf(ws) : -INFINITY;
}

int launch_merge_two(const float* o_a, const float* l_a, const float* o_b, const float* l_b, void* out, int out_bf16,
                     float* lse, long long rows, cudaStream_t stream) {
  if (rows <= 0) return MLA_OK;
  merge_two_kernel<<<static_cast<unsigned>(rows), 128, 0, stream>>>(o_a, l_a, o_b, l_b, out, out_bf16, lse, rows);
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int launch_merge(const MergeParams& p, int entries, int max_pieces, cudaStream_t stream) {
  if (entries <= 0) return MLA_OK;
  const int groups = max_pieces >= 16 ? 4 : max_pieces >= 8 ? 2 : 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(entries, p.heads);
  cfg.blockDim = dim3(128 * groups);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, merge_kernel, p) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // namespace mla
