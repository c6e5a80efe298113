// The two per-head products that put the absorbed decode between the model's
// projections ("MLA and torch.compile: v0.3's two sources", section "MLA:
// starting from a 439-line commit": kv_b_proj is split into w_kc and w_vc;
// decode multiplies q_nope by w_kc before attention and the attention's latent
// output by w_vc after it):
//
//   absorb:   q_nope[b, h, :]  = q_pre[b, h, 0:128]  . w_kc[h]   (w_kc[h]: 128 x 512)
//   project:  out[b, h, :]     = o_lat[b, h, 0:512]  . w_vc[h]   (w_vc[h]: 512 x 128)
//
// Both are C_h = A_h . W_h for every head h, with A_h the rows b of a
// [B, H, K] tensor (row stride H*K) and W_h a row-major K x N matrix.  One CTA
// computes a 128-row x NT-column block of one head on the tensor cores:
//   warp 0   TMA producer: K in chunks of 64, A as K-major 128-byte-swizzled
//            atoms (128 rows x 64), W as N-major atoms (64 K-rows x 64 cols)
//   warp 1   TMEM allocator and MMA issuer: per chunk 4 MMAs M=128, N=NT,
//            K=16 (A K-major, B N-major), accumulator in TMEM
//   warps 4-7  epilogue: TMEM lane = row b, NT fp32 columns converted and
//            stored with 16-byte stores; rows past B (the TMA's zero fill)
//            are not stored
// Every weight byte is read once per 128 requests: the products are batched
// over requests per head, which a per-request decode CTA could not do.
#include <cuda_bf16.h>

#include "mla_device.cuh"
#include "mla_launch.h"

namespace mla {
namespace hg {

constexpr int kThreads = 256;
constexpr int BM = 128, BK = 64;
constexpr int kEpiWarp0 = 4;

template <int K, int N>
struct Cfg {
  static constexpr int NT = N >= 256 ? 256 : N;          // columns per CTA (TMEM columns)
  static constexpr int kChunks = K / BK;
  static constexpr int kStages = kChunks < 3 ? kChunks : 3;
  static constexpr int kABytes = BM * BK * 2;             // 16 KB
  static constexpr int kBBlocks = NT / 64;
  static constexpr int kBBytes = kBBlocks * BK * 128;     // NT x 64 bf16
  static constexpr int kStage = kABytes + kBBytes;
  static constexpr int kOffBar = kStages * kStage;        // full[S], empty[S], done
  static constexpr int kOffMisc = kOffBar + (2 * kStages + 1) * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static constexpr uint32_t kIdesc = idesc_bf16(BM, NT, false, true);
  static_assert(K % BK == 0 && N % NT == 0 && NT % 64 == 0, "tile shape");
  static_assert(kStage % 1024 == 0 && kABytes % 1024 == 0, "atoms must be 1024-byte aligned");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <int K, int N, typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
    head_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                     const HeadGemmParams p) {
  using C = Cfg<K, N>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto full = [&](int s) { return base + C::kOffBar + 8u * s; };
  auto empty = [&](int s) { return base + C::kOffBar + 8u * (C::kStages + s); };
  const uint32_t done = base + C::kOffBar + 16u * C::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const WaitCtx wc{abort_flag, p.status};
  const int n0 = blockIdx.x * C::NT, m0 = blockIdx.y * BM, h = blockIdx.z;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), 1); }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::NT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_w);
      for (int c = 0; c < C::kChunks; ++c) {
        const int s = c % C::kStages;
        if (c >= C::kStages && !mbar_wait(empty(s), ((c / C::kStages) - 1) & 1, wc)) break;
        const uint32_t st = base + s * C::kStage;
        mbar_arrive_expect_tx(full(s), C::kStage);
        tma_load_2d(st, &tm_a, h * K + c * BK, m0, full(s));
#pragma unroll
        for (int j = 0; j < C::kBBlocks; ++j)
          tma_load_2d(st + C::kABytes + j * (BK * 128), &tm_w, n0 + 64 * j, h * K + c * BK, full(s));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      auto D = [](uint64_t d, uint32_t off) -> uint64_t { return d + (off >> 4); };
      bool ok = true;
      for (int c = 0; c < C::kChunks && ok; ++c) {
        const int s = c % C::kStages;
        if (!mbar_wait(full(s), (c / C::kStages) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t st = base + s * C::kStage;
        const uint64_t da = sdesc(st, 16, 1024);                       // A: K-major
        const uint64_t db = sdesc(st + C::kABytes, BK * 128, 1024);    // W: N-major, 64-col blocks
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks)
          umma_ss(tmem, D(da, ks * 32), D(db, ks * 2048), C::kIdesc, (c | ks) != 0 ? 1u : 0u);
        umma_commit(empty(s));
      }
      umma_commit(done);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------- epilogue
    const int q = warp - kEpiWarp0;                  // TMEM lane quadrant (warp % 4)
    const int row = 32 * q + lane, b = m0 + row;
    bool ok = true;
    if (lane == 0) ok = mbar_wait(done, 0, wc);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    tc_fence_after();
    if (ok) {
      OutT* dst = reinterpret_cast<OutT*>(p.out) + (static_cast<size_t>(b) * p.heads + h) * N + n0;
#pragma unroll 1
      for (int c = 0; c < C::NT; c += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + c, v);
        tmem_wait_ld();
        if (b < p.rows) {
          if constexpr (sizeof(OutT) == 2) {
            uint4 w0, w1;
            w0.x = pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1]));
            w0.y = pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3]));
            w0.z = pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5]));
            w0.w = pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7]));
            w1.x = pack_bf16x2(__uint_as_float(v[8]), __uint_as_float(v[9]));
            w1.y = pack_bf16x2(__uint_as_float(v[10]), __uint_as_float(v[11]));
            w1.z = pack_bf16x2(__uint_as_float(v[12]), __uint_as_float(v[13]));
            w1.w = pack_bf16x2(__uint_as_float(v[14]), __uint_as_float(v[15]));
            reinterpret_cast<uint4*>(dst + c)[0] = w0;
            reinterpret_cast<uint4*>(dst + c)[1] = w1;
          } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) d4[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::NT);
}

template <int K, int N, typename OutT>
int launch(const CUtensorMap& tm_a, const CUtensorMap& tm_w, const HeadGemmParams& p, cudaStream_t stream) {
  using C = Cfg<K, N>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(head_gemm_kernel<K, N, OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return MLA_ERR_CUDA;
    attr_done = true;
  }
  const dim3 grid(N / C::NT, (p.rows + BM - 1) / BM, p.heads);
  head_gemm_kernel<K, N, OutT><<<grid, kThreads, C::kSmemBytes, stream>>>(tm_a, tm_w, p);
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace hg

int launch_absorb(const CUtensorMap& tm_a, const CUtensorMap& tm_w, const HeadGemmParams& p, cudaStream_t stream) {
  return hg::launch<128, 512, __nv_bfloat16>(tm_a, tm_w, p, stream);
}

int launch_project(const CUtensorMap& tm_a, const CUtensorMap& tm_w, const HeadGemmParams& p, int out_bf16,
                   cudaStream_t stream) {
  return out_bf16 ? hg::launch<512, 128, __nv_bfloat16>(tm_a, tm_w, p, stream)
                  : hg::launch<512, 128, float>(tm_a, tm_w, p, stream);
}

}  // namespace mla
