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
// A block of 8 warps covers 8 / S heads of one entry; the S warps of a head
// split its partials (warp k takes partials k, k + S, k + 2S, ...), S = 1, 2,
// 4 or 8 from the most pieces an entry has.  A lane owns 16 latent dims (4
// float4 at float4 index 32c + lane of the row, so each load instruction of a
// warp reads 512 contiguous bytes); a warp keeps two partial rows in flight
// while it adds the previous two, and its first two rows are loaded together
// with the LSEs.  A warp's partial LSEs are loaded one per lane, their maximum
// and weights never leave the warp; the S warps of a head are combined in a
// fixed order (each rescaled to the head's maximum) through shared memory.
// The kernel is launched as a programmatic dependent of the decode kernel:
// its blocks are scheduled while the decode kernel drains and wait
// (griddepcontrol.wait) until its partial states are complete and visible.
#include <cuda_bf16.h>

#include "mla_device.cuh"
#include "mla_launch.h"

namespace mla {

constexpr int kMergeWarps = 8;
constexpr int kMergeThreads = 32 * kMergeWarps;

__device__ __forceinline__ void ld_row4(float4 (&v)[4], const float4* src) {
#pragma unroll
  for (int c = 0; c < 4; ++c) v[c] = __ldcg(src + 32 * c);
}
__device__ __forceinline__ void fma_row4(float4 (&acc)[4], float w, const float4 (&v)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    acc[c].x = fmaf(w, v[c].x, acc[c].x);
    acc[c].y = fmaf(w, v[c].y, acc[c].y);
    acc[c].z = fmaf(w, v[c].z, acc[c].z);
    acc[c].w = fmaf(w, v[c].w, acc[c].w);
  }
}
__device__ __forceinline__ void scale_row4(float4 (&acc)[4], float a) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    acc[c].x *= a;
    acc[c].y *= a;
    acc[c].z *= a;
    acc[c].w *= a;
  }
}

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p, const int S) {
  __shared__ float4 s_acc[kMergeWarps][4][32];
  __shared__ float s_m[kMergeWarps], s_ws[kMergeWarps];
  const int e = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = static_cast<int>(blockIdx.y) * (kMergeWarps / S) + warp / S, sub = warp % S;
  // the next kernel in the stream may be scheduled now; it waits for this
  // grid before it touches what this grid reads or writes
  griddep_launch_dependents();
  int b, p0, p1;
  if (p.plan) {
    // device-only plan (graph replays): the entry count, the list and its
    // bounds come from the plan words; the grid covers every possible entry
    const int32_t* hw = p.plan;
    const int W = hw[kHWorkers], n_items = hw[kHItems], n_merges = hw[kHMerges];
    const long long off = kHeaderWords + static_cast<long long>(W) + 1 + 4ll * n_items;
    const bool good = hw[kHMagic] == kPlanMagic && hw[kHVersion] == kPlanVersion && hw[kHHeads] == p.heads &&
                      W == p.workers &&
                      n_items >= 0 && n_merges >= 0 && off + 3ll * n_merges <= p.plan_cap_words;
    if (!good || e >= n_merges) return;
    b = hw[off + 3 * e];
    p0 = hw[off + 3 * e + 1];
    p1 = hw[off + 3 * e + 2];
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
  const bool live = h < H;
  float4 acc[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f, M = -INFINITY;
  if (live) {
    const int n = p1 - p0;
    const int nw = n > sub ? (n - sub + S - 1) / S : 0;     // this warp's partials
    const size_t step = static_cast<size_t>(S) * H * (kLatent / 4);   // float4 between them
    const float4* src = reinterpret_cast<const float4*>(p.part_o + (static_cast<size_t>(p0 + sub) * H + h) * kLatent) +
                        lane;
    float4 va[4], vb[4];
    if (nw > 0) ld_row4(va, src);
    if (nw > 1) ld_row4(vb, src + step);
    for (int c0 = 0; c0 < nw; c0 += 32) {
      const int nc = min(32, nw - c0);
      if (c0 > 0) {
        ld_row4(va, src + c0 * step);
        if (nc > 1) ld_row4(vb, src + (c0 + 1) * step);
      }
      // this chunk's LSEs (one per lane), their maximum, the running state
      const float l = lane < nc ? __ldcg(p.part_lse + static_cast<size_t>(p0 + sub + (c0 + lane) * S) * H + h)
                                : -INFINITY;
      float mc = l;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, off));
      const float mn = fmaxf(M, mc);
      if (mn > -INFINITY && M > -INFINITY && mn != M) {
        const float a = expf(M - mn);
        wsum *= a;
        scale_row4(acc, a);
      }
      M = mn;
      const float wl = (l == -INFINITY || M == -INFINITY) ? 0.f : expf(l - M);
      for (int j = 0; j < nc; j += 2) {
        float4 vc[4], vd[4];
        const bool more = j + 2 < nc;
        if (more) {
          ld_row4(vc, src + (c0 + j + 2) * step);
          if (j + 3 < nc) ld_row4(vd, src + (c0 + j + 3) * step);
        }
        const float w0 = __shfl_sync(0xffffffffu, wl, j);
        const float w1 = __shfl_sync(0xffffffffu, wl, (j + 1) & 31);
        wsum += w0;
        fma_row4(acc, w0, va);
        if (j + 1 < nc) {
          wsum += w1;
          fma_row4(acc, w1, vb);
        }
        if (more) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            va[c] = vc[c];
            vb[c] = vd[c];
          }
        }
      }
    }
  }
  if (S > 1) {
    // the head's S warps, added in a fixed order at the head's maximum
#pragma unroll
    for (int c = 0; c < 4; ++c) s_acc[warp][c][lane] = acc[c];
    if (lane == 0) {
      s_m[warp] = M;
      s_ws[warp] = wsum;
    }
    __syncthreads();
    if (sub != 0 || !live) return;
    float mh = -INFINITY;
    for (int k = 0; k < S; ++k) mh = fmaxf(mh, s_m[warp + k]);
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    wsum = 0.f;
    for (int k = 0; k < S; ++k) {
      const float mk = s_m[warp + k];
      const float a = mk == -INFINITY ? 0.f : expf(mk - mh);
      wsum = fmaf(a, s_ws[warp + k], wsum);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 v = s_acc[warp + k][c][lane];
        acc[c].x = fmaf(a, v.x, acc[c].x);
        acc[c].y = fmaf(a, v.y, acc[c].y);
        acc[c].z = fmaf(a, v.z, acc[c].z);
        acc[c].w = fmaf(a, v.w, acc[c].w);
      }
    }
    M = mh;
  }
  if (!live) return;
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const size_t o = (static_cast<size_t>(b) * H + h) * kLatent;
  if (p.out_bf16) {
    uint2* dst = reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + o) + lane;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[c].x * inv, acc[c].y * inv);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[c].z * inv, acc[c].w * inv);
      dst[32 * c] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
  } else {
    float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o) + lane;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      dst[32 * c] = make_float4(acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv);
  }
  if (lane == 0 && p.lse) p.lse[static_cast<size_t>(b) * H + h] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
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
  // warps per head: a warp takes up to about four partials
  const int S = max_pieces > 16 ? 8 : max_pieces > 8 ? 4 : max_pieces > 4 ? 2 : 1;
  const int heads_per_block = kMergeWarps / S;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(entries, (p.heads + heads_per_block - 1) / heads_per_block);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, merge_kernel, p, S) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // namespace mla
