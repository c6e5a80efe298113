// Absorbed MLA decode for many heads (H = 48..128, step 16) on sm_103a.
//
// With 128 query heads the heads fill the tensor core's 128-row M side, but
// one SM cannot hold the whole problem: the fp32 output O[128 heads x 512]
// alone is all 512 TMEM columns.  So a worker is a cluster of two CTAs that
// split the latent dimensions: CTA c owns latent dims D_c = [256c, 256c+256)
// of every row and half of the rope key.
//
//   QK (per CTA, partial):  S_c[128 h x 64 tok] = Q[:, D_c] . K[:, D_c]^T  (+ its rope half)
//   exchange:               S = S_0 + S_1   (each CTA sends its fp32 partial
//                           to the other through distributed shared memory)
//   softmax:                the same P in both CTAs (identical inputs)
//   PV (per CTA):           O_c[128 h x 256] += P[128 x 64 tok] . V[64 tok x D_c]
//
// so no product is computed twice and no latent byte is loaded twice.
// ("实现差距：MLA 与 DeepSeek V3", section 2.4: s = (s_nope + s_pe) * sm_scale,
// FA2-style online softmax, kv_c reused as the value; "Attention backends",
// paragraph "MLA": every KV byte used by all 128 heads.)
//
// TMEM (512 columns per CTA): O_c [0,256) fp32; the query's latent half
// [256,384) as packed bf16 (A operand of QK, read from TMEM); two score
// buffers [384,448), [448,512).  P (bf16) is written back over the score
// buffer it came from and is the A operand of PV, read from TMEM.
//
// Shared memory per CTA: a ring of 4 latent blocks (64 tokens x 256 dims,
// 32 KB, gathered with TMA gather4), 4 rope atoms (8 KB), the rope query
// (16 KB), the exchange buffer for the peer's partial scores (34 KB) and a
// small ring of slot indices.
//
// Warp roles per CTA (352 threads):
//   warps 0-3   softmax / epilogue; thread h owns head h (TMEM lane h)
//   warp 4      MMA issuer (one thread, event loop)
//   warp 5      TMEM allocator and rope-query loader (TMA)
//   warp 6      index stager (slot numbers to shared memory, L2 row prefetch)
//   warps 7-10  gather producers (every producer takes a slice of every tile)
//
// Softmax per head is thread-local (a head is a TMEM lane), with a lazily
// moved reference maximum (threshold 8 in log2 units) as in the few-heads
// kernel; both CTAs take identical rescale decisions.
#include "mla_device.cuh"
#include "mla_launch.h"

namespace mla {
namespace pair {

constexpr int T = 64;                        // tokens per tile
constexpr int kProducers = 4;
constexpr int kIdxSlots = 4;
constexpr int kProducerWarp0 = 7;
constexpr int kThreads = 32 * (kProducerWarp0 + kProducers);
constexpr int kLatBlocks = 4;                // ring of latent blocks (all producers fill every block)
constexpr int kRopeSlots = 4;
constexpr int kAtom = T * 128;               // 8 KB: 64 tokens x 64 dims
constexpr int kLatBlock = 4 * kAtom;         // 32 KB: 64 tokens x 256 dims
constexpr int kXRow = 64 * 4 + 16;           // exchange row: 64 fp32 + pad (272 B)
constexpr int kOffLat = 0;
constexpr int kOffRope = kOffLat + kLatBlocks * kLatBlock;
constexpr int kOffQR = kOffRope + kRopeSlots * kAtom;   // rope query: 128 rows x 128 B (K-major SW128)
constexpr int kOffX = kOffQR + 128 * 128;
constexpr int kOffIdx = kOffX + 128 * kXRow;
constexpr int kOffBar = kOffIdx + 4 * kIdxSlots * T;
// barriers
constexpr int bLatFull = 0;
constexpr int bLatEmpty = bLatFull + kLatBlocks;
constexpr int bRopeFull = bLatEmpty + kLatBlocks;
constexpr int bRopeEmpty = bRopeFull + kRopeSlots;
constexpr int bQFull = bRopeEmpty + kRopeSlots;
constexpr int bQEmpty = bQFull + 1;
constexpr int bSFull = bQEmpty + 1;          // [2]
constexpr int bPFull = bSFull + 2;           // [2]
constexpr int bSFree = bPFull + 2;           // [2] (PV done with the P in that buffer)
constexpr int bPvDone = bSFree + 2;
constexpr int bOFull = bPvDone + 1;
constexpr int bOEmpty = bOFull + 1;
constexpr int bXFull = bOEmpty + 1;          // peer's partial scores have landed here
constexpr int bXEmpty = bXFull + 1;          // peer has read what this CTA sent
constexpr int bDrain = bXEmpty + 1;
constexpr int bIdxFull = bDrain + 1;
constexpr int bIdxEmpty = bIdxFull + kIdxSlots;
constexpr int kNumBars = bIdxEmpty + kIdxSlots;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffLast = kOffMisc + 16;      // [kLatBlocks + kRopeSlots] last armed use
constexpr int kSmemBytes = kOffLast + 4 * (kLatBlocks + kRopeSlots) + 1024;
constexpr int kTmO = 0, kTmQ = 256, kTmS = 384;
constexpr uint32_t kIdescQK = idesc_bf16(128, T, false, false);     // M=128 heads, N=64 tokens
constexpr uint32_t kIdescPV = idesc_bf16(128, 256, false, true);    // N=256 dims, B (V) MN-major
static_assert(kProducers == 4, "producer pw gathers latent atom pw of the CTA's four");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffRope % 1024 == 0 && kOffQR % 1024 == 0 && kOffX % 16 == 0 && kOffIdx % 16 == 0, "alignment");

__device__ __forceinline__ bool item_ok(const DecodeParams& p, int b, int s, int e) {
  if (b < 0 || b >= p.batch) return false;
  const int lo = __ldg(p.kv_indptr + b), hi = __ldg(p.kv_indptr + b + 1);
  return lo <= s && s < e && e <= hi;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > MLA_WAIT_LIMIT_NS) return;
  }
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  uint32_t a[16];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    tmem_ld16(taddr + 16 * c, a);
#pragma unroll
    for (int i = 0; i < 16; ++i) r[16 * c + i] = a[i];
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    pair_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_qr,
                const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t cta = cluster_ctarank();        // 0 or 1: which latent half
  const uint32_t peer = cta ^ 1u;
  auto bar = [&](int i) -> uint32_t { return base + kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* last_armed = reinterpret_cast<int*>(smem + kOffLast);
  const WaitCtx wc{abort_flag, p.status};

  const int w = blockIdx.x >> 1;
  const int32_t* wptr = p.plan + kHeaderWords;
  const int it0 = wptr[w], it1 = wptr[w + 1];
  const int32_t* items = p.plan + p.items_off;
  const int H = p.heads;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kLatBlocks; ++i) { mbar_init(bar(bLatFull + i), 1); mbar_init(bar(bLatEmpty + i), 1); }
    for (int i = 0; i < kRopeSlots; ++i) { mbar_init(bar(bRopeFull + i), 1); mbar_init(bar(bRopeEmpty + i), 1); }
    mbar_init(bar(bQFull), 5);                   // 4 softmax warps (latent half) + the rope TMA
    mbar_init(bar(bQEmpty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bSFull + i), 1); mbar_init(bar(bPFull + i), 4); mbar_init(bar(bSFree + i), 1);
    }
    mbar_init(bar(bPvDone), 1);
    mbar_init(bar(bOFull), 1);
    mbar_init(bar(bOEmpty), 4);
    mbar_init(bar(bXFull), 1);
    mbar_init(bar(bXEmpty), 4);                  // the peer's four softmax warps
    mbar_init(bar(bDrain), 1);
    for (int i = 0; i < kIdxSlots; ++i) { mbar_init(bar(bIdxFull + i), 1); mbar_init(bar(bIdxEmpty + i), kProducers); }
    for (int i = 0; i < kLatBlocks + kRopeSlots; ++i) last_armed[i] = -1;
    *abort_flag = 0;
    fence_mbar_init();
  }
  // rope-query rows >= H stay zero (the TMA box has H rows)
  for (int i = threadIdx.x; i < (128 * 128) / 16; i += blockDim.x)
    *reinterpret_cast<uint4*>(smem + kOffQR + 16 * i) = make_uint4(0, 0, 0, 0);
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  cluster_sync_all();                            // both CTAs' barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 6) {
    // ---------------------------------------------------------- index stager
    int* idx_ring = reinterpret_cast<int*>(smem + kOffIdx);
    uint32_t g = 0;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
      if (!item_ok(p, b, s, e)) {
        if (lane == 0) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
        continue;
      }
      const int n = e - s;
      for (int t0 = 0; t0 < n; t0 += T, ++g) {
        const uint32_t slot = g % kIdxSlots, use = g / kIdxSlots;
        int v[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) v[k] = __ldg(p.kv_indices + s + min(t0 + lane + 32 * k, n - 1));
        bool w_ok = true;
        if (lane == 0 && use > 0) w_ok = mbar_wait(bar(bIdxEmpty + slot), (use - 1) & 1, wc);
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) { ok = false; break; }
        bool oob = false;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          if (v[k] < 0 || static_cast<long long>(v[k]) >= p.num_slots) { oob = true; v[k] = 0; }
          idx_ring[slot * T + lane + 32 * k] = v[k];
        }
        // this CTA prefetches the lines of every other row into L2
        for (int q = lane; q < 9 * (T / 2); q += 32) {
          const int rr = q / 9, line = q - 9 * rr, r = 2 * rr + static_cast<int>(cta);
          const int lo = __shfl_sync(0xffffffffu, v[0], r & 31);
          const int hi = __shfl_sync(0xffffffffu, v[1], r & 31);
          const int vr = (r >> 5) ? hi : lo;
          if (t0 + r < n) prefetch_l2_line(p.kv_cache + static_cast<size_t>(vr) * (kRow * 2) + line * 128);
        }
        if (__any_sync(0xffffffffu, oob) && lane == 0) record_status(p.status, MLA_ERR_INDEX_OOB);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bIdxFull + slot));
      }
    }
  } else if (warp >= kProducerWarp0) {
    // ------------------------------------------------------ gather producers
    // A warp completes one gather4 only every ~70-110 cycles, so a tile's
    // landing time is set by how many gathers one warp issues for it.  All
    // four producers therefore share every tile: producer pw gathers latent
    // atom pw of the CTA's half (16 gathers) and rope gathers 4pw..4pw+3.
    const int pw = warp - kProducerWarp0;
    if (lane == 0 && pw == 0) tma_prefetch_desc(&tm_kv);
    const uint64_t pol = l2_policy_evict_first();
    const int* idx_ring = reinterpret_cast<const int*>(smem + kOffIdx);
    uint32_t g = 0;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
      if (!item_ok(p, b, s, e)) continue;
      const int n = e - s;
      for (int t0 = 0; t0 < n && ok; t0 += T, ++g) {
        const uint32_t islot = g % kIdxSlots;
        bool w_ok = true;
        if (lane == 0) w_ok = mbar_wait(bar(bIdxFull + islot), (g / kIdxSlots) & 1, wc);
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) { ok = false; break; }
        // lane l < 16 holds tokens 4l..4l+3 (gather op l of an atom)
        const int4 v = *reinterpret_cast<const int4*>(idx_ring + islot * T + 4 * (lane & 15));
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bIdxEmpty + islot));
        if (lane == 0 && pw == 0) MLA_TRACE_EVENT(0, g);
        // rope ops 4pw + r (r = 0..3) take the tokens of op 4pw + r
        const int src = 4 * pw + (lane & 3);
        const int r0 = __shfl_sync(0xffffffffu, v.x, src), r1 = __shfl_sync(0xffffffffu, v.y, src);
        const int r2 = __shfl_sync(0xffffffffu, v.z, src), r3 = __shfl_sync(0xffffffffu, v.w, src);
        // latent atom pw into block g mod 4
        {
          const uint32_t blk = g % kLatBlocks, use = g / kLatBlocks;
          bool e_ok = true;
          if (lane == 0 && use > 0) e_ok = mbar_wait(bar(bLatEmpty + blk), (use - 1) & 1, wc);
          e_ok = __shfl_sync(0xffffffffu, e_ok, 0);
          if (!e_ok) { ok = false; break; }
          const uint32_t full = bar(bLatFull + blk);
          if (lane == 0 && pw == 0) mbar_arrive_expect_tx(full, kLatBlock);
          __syncwarp();
          if (lane < 16)
            tma_gather4(base + kOffLat + blk * kLatBlock + pw * kAtom + lane * 512, &tm_kv,
                        64 * (4 * static_cast<int>(cta) + pw), v.x, v.y, v.z, v.w, full, pol);
          if (lane == 0) atomicMax(last_armed + blk, static_cast<int>(use));
        }
        // rope slice
        {
          const uint32_t rs = g % kRopeSlots, use = g / kRopeSlots;
          bool e_ok = true;
          if (lane == 0 && use > 0) e_ok = mbar_wait(bar(bRopeEmpty + rs), (use - 1) & 1, wc);
          e_ok = __shfl_sync(0xffffffffu, e_ok, 0);
          if (!e_ok) { ok = false; break; }
          const uint32_t full = bar(bRopeFull + rs);
          if (lane == 0 && pw == 0) mbar_arrive_expect_tx(full, kAtom);
          __syncwarp();
          if (lane < 4)
            tma_gather4(base + kOffRope + rs * kAtom + (4 * pw + lane) * 512, &tm_kv, 512, r0, r1, r2, r3, full, pol);
          if (lane == 0) atomicMax(last_armed + kLatBlocks + rs, static_cast<int>(use));
          if (lane == 0 && pw == 0) MLA_TRACE_EVENT(1, g);
        }
      }
    }
    named_bar_sync(3, 32 * kProducers);
    if (pw == 0 && lane < kLatBlocks + kRopeSlots) {
      const int u = last_armed[lane];
      const int bfull = lane < kLatBlocks ? bLatFull + lane : bRopeFull + (lane - kLatBlocks);
      if (u >= 0) drain_wait(bar(bfull), u & 1);
    }
    __syncwarp();
  } else if (warp == 4) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint64_t dk = sdesc(base + kOffLat, 16, 1024);         // latent block 0, K-major (B of QK)
      const uint64_t dv = sdesc(base + kOffLat, kAtom, 1024);      // latent block 0, MN-major (B of PV)
      const uint64_t dr = sdesc(base + kOffRope, 16, 1024);        // rope slot 0 (B of QK)
      const uint64_t dqr = sdesc(base + kOffQR, 16, 1024);         // rope query (A of QK)
      auto D = [](uint64_t d, uint32_t byte_off) -> uint64_t { return d + (byte_off >> 4); };
      const uint32_t bar0 = bar(0);
      auto bar_at = [&](int i) -> uint32_t { return bar0 + 8u * i; };
      auto next_valid = [&](int it) {
        while (it < it1 && !item_ok(p, items[4 * it], items[4 * it + 1], items[4 * it + 2])) ++it;
        return it;
      };
      auto ntiles = [&](int it) { return it < it1 ? (items[4 * it + 2] - items[4 * it + 1] + T - 1) / T : 0; };
      int q_it = next_valid(it0), q_nt = ntiles(q_it), q_j = 0, q_u = 0;
      uint32_t q_g = 0, q_nitem = 0;
      bool q_ready = false;
      int p_it = q_it, p_nt = q_nt, p_j = 0;
      uint32_t p_g = 0, p_nitem = 0;
      uint64_t t_last = globaltimer();
      while (p_it < it1) {
        bool prog = false;
        if (p_g < q_g) {
          const uint32_t buf = p_g & 1;
          const bool first = p_j == 0;
          if (mbar_test_wait(bar_at(bPFull + buf), (p_g >> 1) & 1) &&
              (!first || p_nitem == 0 || mbar_test_wait(bar_at(bOEmpty), (p_nitem - 1) & 1))) {
            tc_fence_after();
            MLA_TRACE_EVENT(4, p_g);
            const uint32_t blk = p_g % kLatBlocks;
            const uint64_t bv = D(dv, blk * kLatBlock);
            const uint32_t a_p = tmem + kTmS + buf * 64;           // P: 64 tokens as 32 packed columns
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_ts(tmem + kTmO, a_p + 8 * ks, D(bv, ks * 2048), kIdescPV, (first && ks == 0) ? 0u : 1u);
            umma_commit(bar_at(bLatEmpty + blk));
            umma_commit(bar_at(bSFree + buf));
            umma_commit(bar_at(bPvDone));
            MLA_TRACE_EVENT(5, p_g);
            if (++p_j == p_nt) {
              umma_commit(bar_at(bOFull));
              ++p_nitem;
              p_it = next_valid(p_it + 1);
              p_nt = ntiles(p_it);
              p_j = 0;
            }
            ++p_g;
            prog = true;
          }
        }
        if (!prog && q_it < it1) {
          if (!q_ready) {
            q_ready = (q_j != 0 || mbar_test_wait(bar_at(bQFull), q_nitem & 1)) &&
                      (q_g < 2 || mbar_test_wait(bar_at(bSFree + (q_g & 1)), ((q_g >> 1) - 1) & 1));
          }
          if (q_ready) {
            const uint32_t d_s = tmem + kTmS + (q_g & 1) * 64;
            if (q_u == 0) {
              const uint32_t blk = q_g % kLatBlocks;
              if (mbar_test_wait(bar_at(bLatFull + blk), (q_g / kLatBlocks) & 1)) {
                tc_fence_after();
                MLA_TRACE_EVENT(2, q_g);
                const uint64_t bk = D(dk, blk * kLatBlock);
#pragma unroll
                for (int k = 0; k < 16; ++k)      // 256 latent dims = 16 K-steps; A (query) from TMEM
                  umma_ts(d_s, tmem + kTmQ + 8 * k, D(bk, (k >> 2) * kAtom + (k & 3) * 32), kIdescQK,
                          k != 0 ? 1u : 0u);
                q_u = 1;
                prog = true;
              }
            } else {
              const uint32_t rs = q_g % kRopeSlots;
              if (mbar_test_wait(bar_at(bRopeFull + rs), (q_g / kRopeSlots) & 1)) {
                tc_fence_after();
                const uint64_t br = D(dr, rs * kAtom);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {  // this CTA's half of the rope dims
                  const uint32_t off = (2 * cta + kk) * 32;
                  umma_ss(d_s, D(dqr, off), D(br, off), kIdescQK, 1u);
                }
                umma_commit(bar_at(bRopeEmpty + rs));
                umma_commit(bar_at(bSFull + (q_g & 1)));
                MLA_TRACE_EVENT(3, q_g);
                const bool last = q_j == q_nt - 1;
                if (last) umma_commit(bar_at(bQEmpty));
                q_u = 0;
                q_ready = false;
                ++q_g;
                if (last) {
                  ++q_nitem;
                  q_it = next_valid(q_it + 1);
                  q_nt = ntiles(q_it);
                  q_j = 0;
                } else {
                  ++q_j;
                }
                prog = true;
              }
            }
          }
        }
        if (prog) {
          t_last = globaltimer();
        } else {
          if (*abort_flag) break;
          if (globaltimer() - t_last > MLA_WAIT_LIMIT_NS) {
            *abort_flag = 1;
            record_status(p.status, MLA_ERR_TIMEOUT);
            break;
          }
        }
      }
      umma_commit(bar_at(bDrain));
      drain_wait(bar_at(bDrain), 0);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------------------------------------------- rope-query loader
    if (lane == 0) {
      tma_prefetch_desc(&tm_qr);
      uint32_t nitem = 0;
      for (int it = it0; it < it1; ++it) {
        const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
        if (!item_ok(p, b, s, e)) continue;
        if (nitem > 0 && !mbar_wait(bar(bQEmpty), (nitem - 1) & 1, wc)) break;
        mbar_arrive_expect_tx(bar(bQFull), H * 128);
        tma_load_2d(base + kOffQR, &tm_qr, 0, b * H, bar(bQFull));
        ++nitem;
      }
      if (nitem > 0) drain_wait(bar(bQFull), (nitem - 1) & 1);
    }
    __syncwarp();
  } else if (warp < 4) {
    // --------------------------------------------------- softmax + epilogue
    const int h = 32 * warp + lane;              // head == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const bool head_ok = h < H;
    const uint32_t x_row = base + kOffX + h * kXRow;                 // my row of the receive buffer
    const uint32_t x_row_peer = mapa_shared(x_row, peer);            // my row in the peer's buffer
    const uint32_t x_full_peer = mapa_shared(bar(bXFull), peer);
    uint32_t g = 0, nitem = 0;
    bool aborted = false;
    float m_ref = 0.f, l_sum = 0.f;
    auto wait = [&](uint32_t bb, uint32_t par, bool cluster_scope) {
      if (aborted) return;
      bool r = true;
      if (lane == 0) r = cluster_scope ? mbar_wait<true>(bb, par, wc) : mbar_wait(bb, par, wc);
      r = __shfl_sync(0xffffffffu, r, 0);
      if (!r) aborted = true;
    };
    for (int it = it0; it < it1; ++it) {
      const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
      const int part = items[4 * it + 3];
      if (!item_ok(p, b, s, e)) continue;
      const int n = e - s, nt = (n + T - 1) / T;
      // -- query latent half into TMEM (after the previous item's last QK)
      if (nitem > 0) wait(bar(bQEmpty), (nitem - 1) & 1, false);
      tc_fence_after();
      if (!aborted) {
        const uint4* src = reinterpret_cast<const uint4*>(p.q_nope + (static_cast<size_t>(b) * H + h) * kLatent +
                                                          256 * cta);
#pragma unroll
        for (int c = 0; c < 8; ++c) {            // 8 x 16 columns = 256 bf16
          uint32_t r[16];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = head_ok ? __ldg(src + 4 * c + k) : make_uint4(0, 0, 0, 0);
            r[4 * k] = v.x; r[4 * k + 1] = v.y; r[4 * k + 2] = v.z; r[4 * k + 3] = v.w;
          }
          tmem_st16(tmem + lane_off + kTmQ + 16 * c, r);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !aborted) mbar_arrive(bar(bQFull));

      // The exchange is software-pipelined: tile j+1's partial row is sent as
      // soon as tile j's has been read, so the transfer runs under tile j's
      // softmax.  `sr` holds this CTA's partial row of the tile in flight.
      uint32_t sr[64];
      auto stage_send = [&](uint32_t gg) {
        const uint32_t tm_s = tmem + lane_off + kTmS + (gg & 1) * 64;
        wait(bar(bSFull + (gg & 1)), (gg >> 1) & 1, false);
        if (threadIdx.x == 0) MLA_TRACE_EVENT(6, gg);
        tc_fence_after();
        if (!aborted) {
          tmem_ld64(tm_s, sr);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) sr[i] = 0;
        }
        if (warp == 0 && lane == 0 && !aborted) mbar_arrive_expect_tx(bar(bXFull), 128 * 64 * 4);
        if (gg > 0) wait(bar(bXEmpty), (gg - 1) & 1, true);      // the peer has read tile gg-1
        if (!aborted) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            st_async_v4(x_row_peer + 16 * i, sr[4 * i], sr[4 * i + 1], sr[4 * i + 2], sr[4 * i + 3], x_full_peer);
        }
      };
      stage_send(g);
      for (int j = 0; j < nt; ++j, ++g) {
        const uint32_t buf = g & 1;
        const uint32_t tm_s = tmem + lane_off + kTmS + buf * 64;
        wait(bar(bXFull), g & 1, true);
        if (threadIdx.x == 0) MLA_TRACE_EVENT(9, g);
        // s = (CTA0 partial + CTA1 partial) in log2 units; the same sum order in both CTAs
        float sv[64];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint4 pv = make_uint4(0, 0, 0, 0);
          if (!aborted)
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(pv.x), "=r"(pv.y), "=r"(pv.z), "=r"(pv.w)
                         : "r"(x_row + 16 * i));
          const uint32_t q[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float own = __uint_as_float(sr[4 * i + k]), oth = __uint_as_float(q[k]);
            sv[4 * i + k] = (cta == 0 ? own + oth : oth + own) * p.scale_log2;
          }
        }
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive_cluster(bar(bXEmpty), peer);   // the peer may send again
        if (j + 1 < nt) stage_send(g + 1);       // next partial goes out while this tile is scored
        const int nvalid = n - j * T;
        if (nvalid < T) {
#pragma unroll
          for (int t = 0; t < 64; ++t)
            if (t >= nvalid) sv[t] = -INFINITY;
        }
        float mt = sv[0];
#pragma unroll
        for (int t = 1; t < 64; ++t) mt = fmaxf(mt, sv[t]);
        if (j == 0) {
          m_ref = mt;
          l_sum = 0.f;
        } else {
          const bool need = mt > m_ref + 8.f;
          if (__any_sync(0xffffffffu, need)) {
            // rescale O (this CTA's 256 dims) after the previous PV has landed
            wait(bar(bPvDone), (g - 1) & 1, false);
            tc_fence_after();
            const float alpha = need ? ex2_approx(m_ref - mt) : 1.f;
            if (need) {
              m_ref = mt;
              l_sum *= alpha;
            }
            if (!aborted) {
#pragma unroll 1
              for (int c = 0; c < 16; ++c) {
                uint32_t o[16];
                tmem_ld16(tmem + lane_off + kTmO + 16 * c, o);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                tmem_st16(tmem + lane_off + kTmO + 16 * c, o);
              }
              tmem_wait_st();
            }
          }
        }
        // P = 2^(s - m_ref) as bf16 pairs over the score buffer
        uint32_t pk[32];
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float a = ex2_approx(sv[2 * i] - m_ref), c = ex2_approx(sv[2 * i + 1] - m_ref);
          l0 += a;
          l1 += c;
          pk[i] = pack_bf16x2(a, c);
        }
        l_sum += l0 + l1;
        if (!aborted) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = pk[16 * c + i];
            tmem_st16(tm_s + 16 * c, r);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(bPFull + buf));
        if (threadIdx.x == 0) MLA_TRACE_EVENT(7, g);
      }
      // ------------------------------------------------------------ epilogue
      wait(bar(bOFull), nitem & 1, false);
      tc_fence_after();
      if (!aborted) {
        const float inv = 1.f / l_sum;
        float* dst_f = nullptr;
        __nv_bfloat16* dst_h = nullptr;
        if (part < 0) {
          const size_t o = (static_cast<size_t>(b) * H + h) * kLatent + 256 * cta;
          if (p.out_bf16) dst_h = reinterpret_cast<__nv_bfloat16*>(p.out) + o;
          else dst_f = reinterpret_cast<float*>(p.out) + o;
        } else {
          dst_f = p.part_o + (static_cast<size_t>(part) * H + h) * kLatent + 256 * cta;
        }
#pragma unroll 1
        for (int c = 0; c < 16; ++c) {
          uint32_t o[16];
          tmem_ld16(tmem + lane_off + kTmO + 16 * c, o);
          tmem_wait_ld();
          if (head_ok) {
            if (dst_f) {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                reinterpret_cast<float4*>(dst_f + 16 * c)[i] =
                    make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
            } else {
              uint32_t hv[8];
#pragma unroll
              for (int i = 0; i < 8; ++i)
                hv[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
              reinterpret_cast<uint4*>(dst_h + 16 * c)[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
              reinterpret_cast<uint4*>(dst_h + 16 * c)[1] = make_uint4(hv[4], hv[5], hv[6], hv[7]);
            }
          }
        }
        if (cta == 0 && head_ok) {
          const float l = (m_ref + __log2f(l_sum)) * 0.69314718055994531f;
          if (part < 0) { if (p.lse) p.lse[static_cast<size_t>(b) * H + h] = l; }
          else p.part_lse[static_cast<size_t>(part) * H + h] = l;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !aborted) mbar_arrive(bar(bOEmpty));
      ++nitem;
    }
    // If this CTA gave up, the peer may still have a partial in flight to us
    // (it sends tile g after we release tile g-1): let it land before exit.
    if (aborted && lane == 0 && warp == 0) drain_wait(bar(bXFull), g & 1);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();                            // no CTA leaves while its peer may still write to it
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
}

}  // namespace pair

int launch_pair(int heads, const CUtensorMap& tm_kv, const CUtensorMap& tm_qn, const CUtensorMap& tm_qr,
                const DecodeParams& p, int workers, cudaStream_t stream) {
  (void)tm_qn;
  if (heads < 48 || heads > 128 || heads % 16 != 0) return MLA_ERR_UNSUPPORTED;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(pair::pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, pair::kSmemBytes) !=
        cudaSuccess)
      return MLA_ERR_CUDA;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * workers, 1, 1);
  cfg.blockDim = dim3(pair::kThreads, 1, 1);
  cfg.dynamicSmemBytes = pair::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, pair::pair_kernel, tm_kv, tm_qr, p) != cudaSuccess) return MLA_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace mla
