// Absorbed MLA decode for few heads (H = 16 or 32) on sm_103a.
//
// With only 16 or 32 query heads the tensor core's 128-row M side cannot be
// the heads, so both products run "swapped": tokens (or latent dims) on M,
// heads on N.
//
//   QK:  S^T[128 tok x H]   = K_tile[128 tok x 576] . Q[H x 576]^T       (K-major A and B)
//   PV:  O^T[128 dim x H]  += V^T[128 dim x 128 tok] . P^T[128 tok x H]   (A read MN-major
//                                                                          from the same tile)
//
// The latent rows are gathered from the page-size-1 cache with TMA gather4
// (four slots per instruction) into 128-byte-swizzled "atoms" of 128 tokens x
// 64 dims (16 KB): 8 latent atoms and 1 rope atom per 128-token tile.  Each
// latent atom is read twice by the tensor core -- once as part of the key
// (score over 576) and once as the value (latent reused as V) -- and leaves
// shared memory after its PV, so every cache byte crosses HBM once.
// ("实现差距：MLA 与 DeepSeek V3", section 2.4: dual-path score, FA2-style
// online softmax, kv_c reused as the value; "Attention backends", paragraph
// "MLA": 576 wide for k and 512 for v, one shared vector per token.)
//
// Warp roles (256 threads, one CTA per SM, persistent over the plan's items):
//   warp 0     gather producer (32 lanes, 4 tokens each, one gather4 per atom)
//   warp 1     MMA issuer (one thread)
//   warp 2     TMEM allocator and query loader (TMA)
//   warps 4-7  softmax / epilogue: thread t owns token row t of S^T and latent
//              row t of every O^T block.
//
// Softmax: scores are scaled into log2 units; each head keeps a reference
// maximum m_ref that only moves when a tile exceeds it by more than 8 (a
// group vote per tile).  Then O and the running sums are rescaled once; so
// P = 2^(s - m_ref) <= 256 always fits bf16 and the fp32 sums.
#include <cstdio>

#include "mla_device.cuh"
#include "mla_launch.h"

namespace mla {
namespace swab {

template <int NH>
struct Cfg {
  static constexpr int T = 128;                    // tokens per tile
  static constexpr int kLatSlots = (NH == 16) ? 10 : 8;  // even: atom pairs never wrap
  static constexpr int kRopeSlots = 2;
  static constexpr int kAtom = T * 128;            // 16 KB
  static constexpr int kQAtom = NH * 128;
  static constexpr int kQBytes = 9 * kQAtom;
  static constexpr int kPAtom = NH * 128;          // NH heads x 64 tokens
  static constexpr int kPBytes = 2 * kPAtom;       // 128 tokens
  static constexpr int kOffLat = 0;
  static constexpr int kOffRope = kOffLat + kLatSlots * kAtom;
  static constexpr int kOffQ = kOffRope + kRopeSlots * kAtom;
  static constexpr int kOffP = kOffQ + kQBytes;
  static constexpr int kOffRed = kOffP + 2 * kPBytes;   // [2][4][NH] floats
  static constexpr int kOffBar = kOffRed + 2 * 4 * NH * 4;
  // barrier indices
  static constexpr int bLatFull = 0;
  static constexpr int bLatEmpty = kLatSlots;
  static constexpr int bRopeFull = 2 * kLatSlots;
  static constexpr int bRopeEmpty = bRopeFull + 2;
  static constexpr int bQFull = bRopeEmpty + 2;
  static constexpr int bQEmpty = bQFull + 1;
  static constexpr int bSFull = bQEmpty + 1;
  static constexpr int bSEmpty = bSFull + 2;
  static constexpr int bPFull = bSEmpty + 2;
  static constexpr int bPEmpty = bPFull + 2;
  static constexpr int bPvDone = bPEmpty + 2;
  static constexpr int bOFull = bPvDone + 1;
  static constexpr int bOEmpty = bOFull + 1;
  static constexpr int bDrain = bOEmpty + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
  static constexpr int kTmemCols = (6 * NH <= 128) ? 128 : 256;
  static constexpr int kTmS = 0;       // S^T buffers: columns [0,NH) and [NH,2NH)
  static constexpr int kTmO = 2 * NH;  // O^T blocks: columns 2NH + mb*NH
  static constexpr uint32_t kIdescQK = idesc_bf16(128, NH, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16(128, NH, true, false);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "atoms must be 1024-byte aligned");
};

__device__ __forceinline__ bool item_ok(const DecodeParams& p, int b, int s, int e) {
  if (b < 0 || b >= p.batch) return false;
  const int lo = __ldg(p.kv_indptr + b), hi = __ldg(p.kv_indptr + b + 1);
  return lo <= s && s < e && e <= hi;
}

// Bounded wait that ignores the abort flag (used to drain in-flight copies).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > MLA_WAIT_LIMIT_NS) return;
  }
}

// Max (or sum) over the 128 softmax threads of v[h], for every h; all threads
// get the result.  `red` is [2][4][NH]; `k` alternates the half in use.
template <int NH, bool kSum>
__device__ __forceinline__ void group_reduce(float (&v)[NH], float* red, int wq, int lane, int& k) {
#pragma unroll
  for (int h = 0; h < NH; ++h) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, v[h], off);
      v[h] = kSum ? v[h] + o : fmaxf(v[h], o);
    }
  }
  float* r = red + (k & 1) * 4 * NH;
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < NH; h += 4)
      *reinterpret_cast<float4*>(r + wq * NH + h) = make_float4(v[h], v[h + 1], v[h + 2], v[h + 3]);
  }
  named_bar_sync(1, 128);
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const float a = r[h], b = r[NH + h], c = r[2 * NH + h], d = r[3 * NH + h];
    v[h] = kSum ? (a + b) + (c + d) : fmaxf(fmaxf(a, b), fmaxf(c, d));
  }
  ++k;
}

template <int NH>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, uint32_t (&r)[NH]) {
  if constexpr (NH == 16) {
    tmem_ld16(taddr, r);
  } else {
    uint32_t a[16], b[16];
    tmem_ld16(taddr, a);
    tmem_ld16(taddr + 16, b);
#pragma unroll
    for (int i = 0; i < 16; ++i) { r[i] = a[i]; r[16 + i] = b[i]; }
  }
}

template <int NH>
__device__ __forceinline__ void tmem_st_row(uint32_t taddr, const uint32_t (&r)[NH]) {
  if constexpr (NH == 16) {
    tmem_st16(taddr, r);
  } else {
    uint32_t a[16], b[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) { a[i] = r[i]; b[i] = r[16 + i]; }
    tmem_st16(taddr, a);
    tmem_st16(taddr + 16, b);
  }
}

template <int NH>
__global__ void __launch_bounds__(256, 1)
    swab_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_qn,
                const __grid_constant__ CUtensorMap tm_qr, const DecodeParams p) {
  using C = Cfg<NH>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return base + C::kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const WaitCtx wc{abort_flag, p.status};

  const int w = blockIdx.x;
  const int32_t* wptr = p.plan + kHeaderWords;
  const int it0 = wptr[w], it1 = wptr[w + 1];
  const int32_t* items = p.plan + p.items_off;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kLatSlots; ++i) { mbar_init(bar(C::bLatFull + i), 1); mbar_init(bar(C::bLatEmpty + i), 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::bRopeFull + i), 1); mbar_init(bar(C::bRopeEmpty + i), 1);
      mbar_init(bar(C::bSFull + i), 1); mbar_init(bar(C::bSEmpty + i), 4);
      mbar_init(bar(C::bPFull + i), 4); mbar_init(bar(C::bPEmpty + i), 1);
    }
    mbar_init(bar(C::bQFull), 1); mbar_init(bar(C::bQEmpty), 1);
    mbar_init(bar(C::bPvDone), 1); mbar_init(bar(C::bOFull), 1); mbar_init(bar(C::bOEmpty), 4);
    mbar_init(bar(C::bDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------- gather producer
    if (lane == 0) { tma_prefetch_desc(&tm_kv); }
    const uint64_t pol = l2_policy_evict_first();
    uint32_t g = 0, lat_issued = 0, rope_issued = 0;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
      if (!item_ok(p, b, s, e)) {
        if (lane == 0) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
        continue;
      }
      const int n = e - s;
      for (int t0 = 0; t0 < n && ok; t0 += C::T, ++g) {
        int y[4];
        bool oob = false;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int tok = min(t0 + 4 * lane + k, n - 1);   // tail rows repeat a valid slot
          int v = __ldg(p.kv_indices + s + tok);
          if (v < 0 || static_cast<long long>(v) >= p.num_slots) { oob = true; v = 0; }
          y[k] = v;
        }
        if (__any_sync(0xffffffffu, oob) && lane == 0) record_status(p.status, MLA_ERR_INDEX_OOB);
        for (int a = 0; a < 9; ++a) {
          uint32_t dst, full, empty, use;
          if (a < 8) {
            const uint32_t seq = g * 8 + a, slot = seq % C::kLatSlots;
            use = seq / C::kLatSlots;
            dst = base + C::kOffLat + slot * C::kAtom;
            full = bar(C::bLatFull + slot);
            empty = bar(C::bLatEmpty + slot);
          } else {
            const uint32_t slot = g & 1;
            use = g >> 1;
            dst = base + C::kOffRope + slot * C::kAtom;
            full = bar(C::bRopeFull + slot);
            empty = bar(C::bRopeEmpty + slot);
          }
          bool w_ok = true;
          if (lane == 0 && use > 0) w_ok = mbar_wait(empty, (use - 1) & 1, wc);
          w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
          if (!w_ok) { ok = false; break; }
          if (lane == 0) mbar_arrive_expect_tx(full, C::kAtom);
          __syncwarp();
          tma_gather4(dst + lane * 512, &tm_kv, 64 * a, y[0], y[1], y[2], y[3], full, pol);
          if (a < 8) ++lat_issued; else ++rope_issued;
        }
      }
    }
    // drain: wait for the last armed phase of every slot (in-flight copies)
    if (lane == 0) {
      for (uint32_t s = 0; s < (uint32_t)C::kLatSlots; ++s)
        if (lat_issued > s) drain_wait(bar(C::bLatFull + s), ((lat_issued - 1 - s) / C::kLatSlots) & 1);
      for (uint32_t s = 0; s < 2; ++s)
        if (rope_issued > s) drain_wait(bar(C::bRopeFull + s), ((rope_issued - 1 - s) / 2) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t g = 0, nitem = 0;
      bool ok = true;
      const uint32_t qbase = base + C::kOffQ;
      auto issue_pv = [&](uint32_t gp, bool first) -> bool {
        const uint32_t buf = gp & 1;
        if (!mbar_wait(bar(C::bPFull + buf), (gp >> 1) & 1, wc)) return false;
        if (first && nitem > 0 && !mbar_wait(bar(C::bOEmpty), (nitem - 1) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t lat0 = (gp * 8) % C::kLatSlots;
        const uint32_t pbase = base + C::kOffP + buf * C::kPBytes;
#pragma unroll 1
        for (int mb = 0; mb < 4; ++mb) {
          const uint32_t slot = (lat0 + 2 * mb) % C::kLatSlots;
          const uint32_t a_addr = base + C::kOffLat + slot * C::kAtom;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t ad = sdesc(a_addr + ks * 2048, C::kAtom, 1024);
            const uint64_t bd = sdesc(pbase + (ks >> 2) * C::kPAtom + (ks & 3) * 32, 16, 1024);
            umma_ss(tmem + C::kTmO + mb * NH, ad, bd, C::kIdescPV, (first && ks == 0) ? 0u : 1u);
          }
          umma_commit(bar(C::bLatEmpty + slot));
          umma_commit(bar(C::bLatEmpty + slot + 1));
        }
        umma_commit(bar(C::bPEmpty + buf));
        umma_commit(bar(C::bPvDone));
        return true;
      };
      // PV of a tile is issued after the QK of the next one (so the softmax
      // overlaps that QK), or earlier if that QK needs a ring slot the PV frees.
      int64_t pending = -1;        // tile whose PV is not issued yet
      bool pending_first = false;
      for (int it = it0; it < it1 && ok; ++it) {
        const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
        if (!item_ok(p, b, s, e)) continue;
        const int nt = (e - s + C::T - 1) / C::T;
        if (!mbar_wait(bar(C::bQFull), nitem & 1, wc)) { ok = false; break; }
        tc_fence_after();
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t buf = g & 1;
          if (g >= 2 && !mbar_wait(bar(C::bSEmpty + buf), ((g >> 1) - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_s = tmem + C::kTmS + buf * NH;
          for (int a = 0; a < 9; ++a) {
            uint32_t src, full, use;
            if (a < 8) {
              const uint32_t seq = g * 8 + a, slot = seq % C::kLatSlots;
              use = seq / C::kLatSlots;
              src = base + C::kOffLat + slot * C::kAtom;
              full = bar(C::bLatFull + slot);
              if (pending >= 0 && seq >= (uint32_t)C::kLatSlots &&
                  (seq - C::kLatSlots) / 8 == static_cast<uint32_t>(pending)) {
                if (!issue_pv(static_cast<uint32_t>(pending), pending_first)) { ok = false; break; }
                pending = -1;
              }
            } else {
              src = base + C::kOffRope + (g & 1) * C::kAtom;
              use = g >> 1;
              full = bar(C::bRopeFull + (g & 1));
            }
            if (!mbar_wait(full, use & 1, wc)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = sdesc(src + 32 * kk, 16, 1024);
              const uint64_t bd = sdesc(qbase + a * C::kQAtom + 32 * kk, 16, 1024);
              umma_ss(d_s, ad, bd, C::kIdescQK, (a | kk) != 0 ? 1u : 0u);
            }
          }
          if (!ok) break;
          umma_commit(bar(C::bSFull + buf));
          umma_commit(bar(C::bRopeEmpty + (g & 1)));
          if (j == nt - 1) umma_commit(bar(C::bQEmpty));
          if (pending >= 0 && !issue_pv(static_cast<uint32_t>(pending), pending_first)) { ok = false; break; }
          pending = g;
          pending_first = (j == 0);
        }
        if (!ok) break;
        if (!issue_pv(static_cast<uint32_t>(pending), pending_first)) { ok = false; break; }
        pending = -1;
        umma_commit(bar(C::bOFull));
        ++nitem;
      }
      // every MMA issued by this thread has completed before TMEM is freed
      umma_commit(bar(C::bDrain));
      drain_wait(bar(C::bDrain), 0);
    }
    __syncwarp();
  } else if (warp == 2) {
    // --------------------------------------------------------- query loader
    if (lane == 0) {
      tma_prefetch_desc(&tm_qn);
      tma_prefetch_desc(&tm_qr);
      uint32_t nitem = 0;
      const uint32_t qbase = base + C::kOffQ;
      for (int it = it0; it < it1; ++it) {
        const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
        if (!item_ok(p, b, s, e)) continue;
        if (nitem > 0 && !mbar_wait(bar(C::bQEmpty), (nitem - 1) & 1, wc)) break;
        mbar_arrive_expect_tx(bar(C::bQFull), C::kQBytes);
        for (int a = 0; a < 8; ++a) tma_load_2d(qbase + a * C::kQAtom, &tm_qn, 64 * a, b * p.heads, bar(C::bQFull));
        tma_load_2d(qbase + 8 * C::kQAtom, &tm_qr, 0, b * p.heads, bar(C::bQFull));
        ++nitem;
      }
      if (nitem > 0) drain_wait(bar(C::bQFull), (nitem - 1) & 1);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // --------------------------------------------------- softmax + epilogue
    const int t = threadIdx.x - 128;   // token row of S^T; latent row of O^T
    const int wq = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    float* red = reinterpret_cast<float*>(smem + C::kOffRed);
    int rk = 0;
    uint32_t g = 0, nitem = 0;
    bool aborted = false;
    float m_ref[NH], l_part[NH];
    auto wait = [&](uint32_t bb, uint32_t par) {
      if (aborted) return;
      bool r = true;
      if (lane == 0) r = mbar_wait(bb, par, wc);
      r = __shfl_sync(0xffffffffu, r, 0);
      if (!r) aborted = true;
    };
    for (int it = it0; it < it1; ++it) {
      const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
      const int part = items[4 * it + 3];
      if (!item_ok(p, b, s, e)) continue;
      const int n = e - s, nt = (n + C::T - 1) / C::T;
      for (int j = 0; j < nt; ++j, ++g) {
        const uint32_t buf = g & 1;
        wait(bar(C::bSFull + buf), (g >> 1) & 1);
        tc_fence_after();
        uint32_t r[NH];
        if (!aborted) {
          tmem_ld_row<NH>(tmem + lane_off + C::kTmS + buf * NH, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int h = 0; h < NH; ++h) r[h] = 0;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(C::bSEmpty + buf));
        const bool valid = t < n - j * C::T;
        float sv[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) sv[h] = valid ? __uint_as_float(r[h]) * p.scale_log2 : -INFINITY;
        if (j == 0) {
#pragma unroll
          for (int h = 0; h < NH; ++h) { m_ref[h] = sv[h]; l_part[h] = 0.f; }
          group_reduce<NH, false>(m_ref, red, wq, lane, rk);
        } else {
          bool need = false;
#pragma unroll
          for (int h = 0; h < NH; ++h) need |= sv[h] > m_ref[h] + 8.f;
          need = named_bar_or(2, 128, need);
          if (need) {
            float mt[NH], alpha[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) mt[h] = sv[h];
            group_reduce<NH, false>(mt, red, wq, lane, rk);
#pragma unroll
            for (int h = 0; h < NH; ++h) {
              const float mn = fmaxf(m_ref[h], mt[h]);
              alpha[h] = ex2_approx(m_ref[h] - mn);
              m_ref[h] = mn;
              l_part[h] *= alpha[h];
            }
            // rescale O^T after the previous tile's PV has landed
            wait(bar(C::bPvDone), (g - 1) & 1);
            tc_fence_after();
            if (!aborted) {
#pragma unroll 1
              for (int mb = 0; mb < 4; ++mb) {
                uint32_t o[NH];
                const uint32_t ta = tmem + lane_off + C::kTmO + mb * NH;
                tmem_ld_row<NH>(ta, o);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < NH; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
                tmem_st_row<NH>(ta, o);
              }
              tmem_wait_st();
            }
          }
        }
        float pv[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          pv[h] = ex2_approx(sv[h] - m_ref[h]);   // -inf rows give 0
          l_part[h] += pv[h];
        }
        if (g >= 2) wait(bar(C::bPEmpty + buf), ((g >> 1) - 1) & 1);
        if (!aborted) {
          // P^T[buf]: K-major, 128B swizzle; row = head, 64 tokens per 128-byte row
          uint8_t* pb = smem + C::kOffP + buf * C::kPBytes + (t >> 6) * C::kPAtom;
          const int tw = t & 63;
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const int off = (h >> 3) * 1024 + (h & 7) * 128 + ((((tw >> 3) ^ (h & 7)) & 7) << 4) + (tw & 7) * 2;
            *reinterpret_cast<__nv_bfloat16*>(pb + off) = __float2bfloat16_rn(pv[h]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(C::bPFull + buf));
      }
      // ------------------------------------------------------------ epilogue
      wait(bar(C::bOFull), nitem & 1);
      tc_fence_after();
      float l_tot[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) l_tot[h] = l_part[h];
      group_reduce<NH, true>(l_tot, red, wq, lane, rk);
      if (!aborted) {
#pragma unroll 1
        for (int mb = 0; mb < 4; ++mb) {
          uint32_t o[NH];
          tmem_ld_row<NH>(tmem + lane_off + C::kTmO + mb * NH, o);
          tmem_wait_ld();
          const int dim = 128 * mb + t;
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const float v = __uint_as_float(o[h]) / l_tot[h];
            if (part < 0) {
              const size_t idx = (static_cast<size_t>(b) * p.heads + h) * kLatent + dim;
              if (p.out_bf16) reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
              else reinterpret_cast<float*>(p.out)[idx] = v;
            } else {
              p.part_o[(static_cast<size_t>(part) * p.heads + h) * kLatent + dim] = v;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !aborted) mbar_arrive(bar(C::bOEmpty));
      if (!aborted) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          if (t == h) {
            const float l = (m_ref[h] + __log2f(l_tot[h])) * 0.69314718055994531f;
            if (part < 0) { if (p.lse) p.lse[static_cast<size_t>(b) * p.heads + h] = l; }
            else p.part_lse[static_cast<size_t>(part) * p.heads + h] = l;
          }
        }
      }
      ++nitem;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, C::kTmemCols);
}

template <int NH>
int launch(const CUtensorMap& tm_kv, const CUtensorMap& tm_qn, const CUtensorMap& tm_qr,
           const DecodeParams& p, int grid, cudaStream_t stream) {
  using C = Cfg<NH>;
  static bool attr_done = false;   // per process; the attribute is per function
  if (!attr_done) {
    if (cudaFuncSetAttribute(swab_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return MLA_ERR_CUDA;
    attr_done = true;
  }
  swab_kernel<NH><<<grid, 256, C::kSmemBytes, stream>>>(tm_kv, tm_qn, tm_qr, p);
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace swab

int launch_swab(int heads, const CUtensorMap& tm_kv, const CUtensorMap& tm_qn,
                const CUtensorMap& tm_qr, const DecodeParams& p, int grid, cudaStream_t stream) {
  if (heads == 16) return swab::launch<16>(tm_kv, tm_qn, tm_qr, p, grid, stream);
  if (heads == 32) return swab::launch<32>(tm_kv, tm_qn, tm_qr, p, grid, stream);
  return MLA_ERR_UNSUPPORTED;
}

int swab_tile_tokens() { return swab::Cfg<16>::T; }

}  // namespace mla
