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
// [B, H, K] tensor (row stride H*K) and W_h a row-major K x N matrix.  A tile
// is a 128-row x NT-column block of one head; one CTA per SM walks the tiles:
//   warp 0   TMA producer: K in chunks of 64, A as K-major 128-byte-swizzled
//            atoms (128 rows x 64), W as N-major atoms (64 K-rows x 64 cols)
//   warp 1   TMEM allocator and MMA issuer: per chunk 4 MMAs M=128, N=NT,
//            K=16 (A K-major, B N-major), two TMEM accumulators in turn
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

// L2 prefetch of one box of a tiled tensor map (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
}

constexpr int kThreads = 256;
constexpr int BM = 128, BK = 64;
constexpr int kEpiWarp0 = 4;
#ifndef MLA_HG_ABSORB_COLS
#define MLA_HG_ABSORB_COLS 64
#endif
#ifndef MLA_HG_PROJECT_COLS
#define MLA_HG_PROJECT_COLS 64
#endif
// Columns per tile: narrower tiles give more tiles to spread over the SMs at
// small batch sizes (the A rows are then re-read from L2 per column block).
constexpr int kAbsorbCols = MLA_HG_ABSORB_COLS, kProjectCols = MLA_HG_PROJECT_COLS;

template <int K, int N, int NT_>
struct Cfg {
  static constexpr int NT = NT_;                          // columns per tile (TMEM columns per accumulator)
  static constexpr int kChunks = K / BK;                  // K chunks per tile
  static constexpr int kABytes = BM * BK * 2;             // 16 KB
  static constexpr int kBBlocks = NT / 64;
  static constexpr int kBBytes = kBBlocks * BK * 128;     // 64 K-rows x NT bf16
  static constexpr int kStage = kABytes + kBBytes;
  static constexpr int kStages = (200 * 1024) / kStage < 6 ? (200 * 1024) / kStage : 6;
  static constexpr int kOffBar = kStages * kStage;        // full[S], empty[S], acc_full[2], acc_empty[2]
  static constexpr int kOffMisc = kOffBar + (2 * kStages + 4) * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static constexpr int kTmemCols = 2 * NT;                // two accumulators
  static constexpr uint32_t kIdesc = idesc_bf16(BM, NT, false, true);
  static_assert(K % BK == 0 && N % NT == 0 && NT % 64 == 0 && kStages >= 2, "tile shape");
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation");
  static_assert(kStage % 1024 == 0 && kABytes % 1024 == 0, "atoms must be 1024-byte aligned");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Persistent: CTA c takes tiles c, c + gridDim.x, ... (tile = (head, 128-row
// block, NT-column block), column block fastest so neighbours share A rows in
// L2).  The producer streams K chunks of consecutive tiles through one ring;
// the MMA issuer alternates two TMEM accumulators, so the epilogue of one tile
// overlaps the loads and MMAs of the next.
template <int K, int N, int NT, typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
    head_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                     const HeadGemmParams p) {
  using C = Cfg<K, N, NT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto full = [&](int s) { return base + C::kOffBar + 8u * s; };
  auto empty = [&](int s) { return base + C::kOffBar + 8u * (C::kStages + s); };
  auto acc_full = [&](int i) { return base + C::kOffBar + 8u * (2 * C::kStages + i); };
  auto acc_empty = [&](int i) { return base + C::kOffBar + 8u * (2 * C::kStages + 2 + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const WaitCtx wc{abort_flag, p.status};
  constexpr int kColTiles = N / NT;
  const int row_tiles = (p.rows + BM - 1) / BM;
  const int tiles = p.heads * row_tiles * kColTiles;
  auto tile_of = [&](int t, int& h, int& m0, int& n0) {
    n0 = (t % kColTiles) * NT;
    m0 = ((t / kColTiles) % row_tiles) * BM;
    h = t / (kColTiles * row_tiles);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(acc_full(i), 1); mbar_init(acc_empty(i), 4); }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // While the previous kernel drains, this CTA's first two tiles (weights and
  // rows) are prefetched into L2.  Only prefetched: the rows may still be
  // written by that kernel, and L2 is where every write lands, so the loads
  // after the wait below still see the final data; the prefetch only takes
  // the DRAM latency off the chain that follows the wait.
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_w);
    for (int t = blockIdx.x, n = 0; t < tiles && n < 2; t += gridDim.x, ++n) {
      int h, m0, n0;
      tile_of(t, h, m0, n0);
      for (int k = 0; k < C::kChunks; ++k) {
        tma_prefetch_l2_2d(&tm_a, h * K + k * BK, m0);
#pragma unroll
        for (int j = 0; j < C::kBBlocks; ++j) tma_prefetch_l2_2d(&tm_w, n0 + 64 * j, h * K + k * BK);
      }
    }
  }
  // a programmatic dependent of the previous kernel in the stream (the setup
  // above overlapped its tail): its results are read only once it has
  // finished; the next kernel may be scheduled from here on
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t c = 0;                              // chunk count over all tiles
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        int h, m0, n0;
        tile_of(t, h, m0, n0);
        for (int k = 0; k < C::kChunks; ++k, ++c) {
          const uint32_t s = c % C::kStages;
          if (c >= static_cast<uint32_t>(C::kStages) &&
              !mbar_wait(empty(s), ((c / C::kStages) - 1) & 1, wc)) { ok = false; break; }
          const uint32_t st = base + s * C::kStage;
          mbar_arrive_expect_tx(full(s), C::kStage);
          tma_load_2d(st, &tm_a, h * K + k * BK, m0, full(s));
#pragma unroll
          for (int j = 0; j < C::kBBlocks; ++j)
            tma_load_2d(st + C::kABytes + j * (BK * 128), &tm_w, n0 + 64 * j, h * K + k * BK, full(s));
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      auto D = [](uint64_t d, uint32_t off) -> uint64_t { return d + (off >> 4); };
      uint32_t c = 0, i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++i) {
        const uint32_t buf = i & 1;
        // the epilogue has read this accumulator's previous tile
        if (i >= 2 && !mbar_wait(acc_empty(buf), ((i >> 1) - 1) & 1, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * NT;
        for (int k = 0; k < C::kChunks; ++k, ++c) {
          const uint32_t s = c % C::kStages;
          if (!mbar_wait(full(s), (c / C::kStages) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = base + s * C::kStage;
          const uint64_t da = sdesc(st, 16, 1024);                       // A: K-major
          const uint64_t db = sdesc(st + C::kABytes, BK * 128, 1024);    // W: N-major, 64-col blocks
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            umma_ss(d, D(da, ks * 32), D(db, ks * 2048), C::kIdesc, (k | ks) != 0 ? 1u : 0u);
          umma_commit(empty(s));
        }
        if (ok) umma_commit(acc_full(buf));
      }
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------- epilogue
    const int q = warp - kEpiWarp0;                  // TMEM lane quadrant (warp % 4)
    const int row = 32 * q + lane;
    uint32_t i = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
      int h, m0, n0;
      tile_of(t, h, m0, n0);
      const uint32_t buf = i & 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(acc_full(buf), (i >> 1) & 1, wc);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int b = m0 + row;
      OutT* dst = reinterpret_cast<OutT*>(p.out) + (static_cast<size_t>(b) * p.heads + h) * N + n0;
#pragma unroll 1
      for (int c = 0; c < NT; c += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * NT + c, v);
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
            for (int j = 0; j < 4; ++j) d4[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(buf));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

template <int K, int N, int NT, typename OutT>
int launch(const CUtensorMap& tm_a, const CUtensorMap& tm_w, const HeadGemmParams& p, cudaStream_t stream) {
  using C = Cfg<K, N, NT>;
  if (!set_smem_limit(reinterpret_cast<const void*>(&head_gemm_kernel<K, N, NT, OutT>), C::kSmemBytes))
    return MLA_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms < 1) return MLA_ERR_CUDA;
  const int tiles = p.heads * ((p.rows + BM - 1) / BM) * (N / C::NT);
  const int grid = tiles < sms ? tiles : sms;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // setup overlaps the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, head_gemm_kernel<K, N, NT, OutT>, tm_a, tm_w, p) != cudaSuccess) return MLA_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace hg

int launch_absorb(const CUtensorMap& tm_a, const CUtensorMap& tm_w, const HeadGemmParams& p, cudaStream_t stream) {
  return hg::launch<128, 512, hg::kAbsorbCols, __nv_bfloat16>(tm_a, tm_w, p, stream);
}

int launch_project(const CUtensorMap& tm_a, const CUtensorMap& tm_w, const HeadGemmParams& p, int out_bf16,
                   cudaStream_t stream) {
  return out_bf16 ? hg::launch<512, 128, hg::kProjectCols, __nv_bfloat16>(tm_a, tm_w, p, stream)
                  : hg::launch<512, 128, hg::kProjectCols, float>(tm_a, tm_w, p, stream);
}

}  // namespace mla
