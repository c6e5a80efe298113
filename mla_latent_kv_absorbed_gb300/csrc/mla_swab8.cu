// Absorbed MLA decode over an FP8 (E4M3) latent cache for few heads (H = 16
// or 32) on sm_103a, with the 8-bit cache bytes fed straight to the tensor
// core (tcgen05.mma kind::f8f6f4) -- no dequantisation pass.
// ("MLA and torch.compile: v0.3's two sources", section "MLA: starting from a
// 439-line commit": the FP8 KV cache is one of the four parts of the 3-7x;
// "实现差距：MLA 与 DeepSeek V3", section 2.4: dual-path score, FA2-style
// online softmax, kv_c reused as the value, FP8 packing of the cache.)
//
// A cache row is 576 E4M3 codes (latent, then rope key); its values are the
// codes times kv_scale (one float32 for the whole cache).  The query and the
// softmax weights are bf16-precise and the tensor core takes two 8-bit
// operands, so each is carried as two E4M3 parts, hi + lo / 32:
//   query (per request and head, by the prep kernel): q' = q * 2^a with a
//     power of two a that puts max |q'| in [128, 256); hi = e4m3(q'),
//     lo = e4m3((q' - hi) * 32).  hi + lo / 32 holds q' to 8 significant bits
//     (bf16 has 8), exactly for |q'| >= 2^-7.
//   weights (per tile, by the softmax warps): P = 2^(s - m_ref) <= 256,
//     hi = e4m3(P), lo = e4m3((P - hi) * 32); relative error <= 2^-8, the same
//     bound as rounding P to bf16.  The running sums add hi + lo / 32, so the
//     normalisation matches the weights the MMA used.
// The two parts ride along N of the same MMA (hi and lo rows of B), so they
// cost no extra instructions; the sum hi + lo / 32 is taken in fp32 when the
// accumulators are read.
//
// Tile (64 tokens), folded like the bf16 kernel: score dims split in halves
//   h0 = latent 0-255 + rope 0-31,  h1 = latent 256-511 + rope 32-63,
// stacked on M:  S[128 x 4H] = [K_h0; K_h1] . [Qhi_h0; Qhi_h1; Qlo_h0; Qlo_h1]^T,
// 8 latent K-steps of 32 dims + 1 rope K-step = 9 MMAs (rows 0-63 x cols
// [0,H) + [2H,3H) are the h0 partials, rows 64-127 x [H,2H) + [3H,4H) the h1).
// PV: O^T[128 dims x 2H] += V^T[128 x 64 tok] . [Phi; Plo]^T, A read MN-major
// from the same atoms, 4 blocks x 2 K-steps = 8 MMAs.  17 MMAs a tile against
// the bf16 kernel's 34, and half the bytes.
//
// Shared-memory unit of one tile (36 KB), filled by TMA gather4:
//   [atom0 | atom2 | atom1 | atom3]   64 tok x 128 dims each, 128-B swizzle
//   [R0 | R1]                         64 tok x 32 rope dims each, 32-B swizzle
// atom c+2 follows atom c so one 128-row descriptor covers both halves; R1 is
// the rope from dim 544 (the h1 rope at K offset 0).
//
// Warp roles (one CTA per SM, persistent over the plan's work items):
//   warps 0-3   softmax / epilogue (TMEM lane quadrants 0-3)
//   warp 4      QK issuer and query-image loader
//   warp 5      TMEM allocator and PV issuer
//   warps 6-13  gather producers: token half j >> 2, latent atom j & 3 (8
//               gather4 of 128-B rows) plus four gather4 of the rope
//
// The prep kernel writes each request's query image (the B operand of QK, in
// its shared-memory byte order) and per-head factors 2^-a to the workspace;
// this kernel is launched as its programmatic dependent, so the gathers of
// the first tiles overlap it, and only the QK and softmax warps wait for it.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "mla_device.cuh"
#include "mla_launch.h"

namespace mla {
namespace swab8 {

constexpr int T = 64;                      // tokens per tile
constexpr int kQkWarp = 4, kPvWarp = 5, kProducerWarp0 = 6;
constexpr int kProducers = 8;
constexpr int kThreads = 32 * (kProducerWarp0 + kProducers);   // 448
constexpr int kAtom = T * 128;             // 8 KB
constexpr int kRopeAtom = T * 32;          // 2 KB
constexpr int kUnit = 4 * kAtom + 2 * kRopeAtom;
constexpr int kRopeOff = 4 * kAtom;
constexpr float kLoWeight = 1.f / 32.f;    // value of a lo part relative to its hi part
#ifndef MLA_SWAB8_LEAD
#define MLA_SWAB8_LEAD 3
#endif
// a producer issues unit g's gathers only once unit g - kLead has landed
constexpr int kLead = MLA_SWAB8_LEAD;
constexpr int kBarSm = 1, kBarVote = 2, kBarPair0 = 3, kBarProd = 5;   // named barriers

// position of latent atom a (dims 128a..) inside a unit
__host__ __device__ constexpr int atom_pos(int a) { return ((a & 1) << 1) | (a >> 1); }

template <int NH>
struct Cfg {
  static constexpr int kHalf = NH / 2;
  static constexpr int kUnits = (NH == 16) ? 5 : 4;
  static_assert(kLead <= kUnits, "a unit's phase must not be lapped while it is waited on");
  static constexpr int kR128 = 4 * NH * 128;            // one 128-dim column of the query image
  static constexpr int kImg = 4 * NH * 288;             // query image of one request
  static constexpr int kPBuf = 2 * NH * 128;            // [Phi; Plo]^T: 2NH rows x 64 tokens (128-B rows)
  static constexpr int kXBytes = 2 * kHalf * T * 4;
  static constexpr int kStage = NH * 128 * 4;
  static constexpr int kOffUnit = 0;
  static constexpr int kOffQ = kUnits * kUnit;
  static constexpr int kOffP = kOffQ + kImg;
  static constexpr int kOffX = kOffP + 2 * kPBuf;
  static constexpr int kOffRed = kOffX + kStage;
  static constexpr int kOffBc = kOffRed + 8 * kHalf * 4;
  static constexpr int bFull = 0;
  static constexpr int bEmpty = bFull + kUnits;
  static constexpr int bQFull = bEmpty + kUnits;
  static constexpr int bQEmpty = bQFull + 1;
  static constexpr int bSFull = bQEmpty + 1;            // [2]
  static constexpr int bSEmpty = bSFull + 2;            // [2]
  static constexpr int bPFull = bSEmpty + 2;            // [2]
  static constexpr int bPDone = bPFull + 2;             // [2]
  static constexpr int bOBlk = bPDone + 2;              // [2] an item's PVs of blocks 0-1 / 2-3 are done
  static constexpr int bOEmpty = bOBlk + 2;
  static constexpr int bDrain = bOEmpty + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kOffBar = kOffBc + NH * 4;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffLast = kOffMisc + 32;
  static constexpr int kSmemBytes = kOffLast + 4 * kUnits + 1024;
  static constexpr int kTmemCols = (NH == 16) ? 256 : 512;
  static constexpr int kTmS = 0;                        // 2 x 4NH
  static constexpr int kTmO = 8 * NH;                   // 4 blocks x 2NH (hi, lo)
  static constexpr uint32_t kIdescQK = idesc_e4m3(128, 4 * NH, false, false);
  static constexpr uint32_t kIdescPV = idesc_e4m3(128, 2 * NH, true, false);
  static_assert(kStage >= kXBytes, "the exchange and the epilogue staging share a region");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kPBuf % 1024 == 0 && kImg % 1024 == 0 && kUnit % 1024 == 0,
                "atoms must be 1024-byte aligned");
  static_assert(kTmO + 8 * NH <= kTmemCols, "TMEM budget");
};

__device__ __forceinline__ bool item_ok(const DecodeParams& p, int nnz, int b, int s, int e) {
  return b >= 0 && b < p.batch && 0 <= s && s < e && e <= nnz;
}
__device__ __forceinline__ bool item_in_request(const DecodeParams& p, int b, int s, int e) {
  const int lo = __ldg(p.kv_indptr + b), hi = __ldg(p.kv_indptr + b + 1);
  return lo <= s && e <= hi;
}
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > MLA_WAIT_LIMIT_NS) return;
  }
}

// Max (or sum) over the two warps of a pair of v[i] for every i (both warps
// get the result); `red` is [2 bufs][2 pairs][2 warps][K].
template <int K, bool kSum>
__device__ __forceinline__ void pair_reduce(float (&v)[K], float* red, int pair, int wip, int lane, int& k) {
#pragma unroll
  for (int i = 0; i < K; ++i) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], off);
      v[i] = kSum ? v[i] + o : fmaxf(v[i], o);
    }
  }
  float* r = red + ((k & 1) * 2 + pair) * 2 * K;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < K; i += 4)
      *reinterpret_cast<float4*>(r + wip * K + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
  }
  named_bar_sync(kBarPair0 + pair, 64);
#pragma unroll
  for (int i = 0; i < K; ++i) v[i] = kSum ? r[i] + r[K + i] : fmaxf(r[i], r[K + i]);
  ++k;
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
#pragma unroll
  for (int c = 0; c < N / 16; ++c) {
    uint32_t a[16];
    tmem_ld16(taddr + 16 * c, a);
#pragma unroll
    for (int i = 0; i < 16; ++i) r[16 * c + i] = a[i];
  }
}

template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
#pragma unroll
  for (int c = 0; c < N / 16; ++c) {
    uint32_t a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = r[16 * c + i];
    tmem_st16(taddr + 16 * c, a);
  }
}

// Byte offset of row n, byte k (< 128) in a 128-byte-swizzled K-major operand.
__host__ __device__ __forceinline__ uint32_t sw128_off(int n, int k) {
  return (n >> 3) * 1024 + (n & 7) * 128 + ((((k >> 4) ^ (n & 7)) & 7) << 4) + (k & 15);
}
// Byte offset of row n, byte k (< 32) in a 32-byte-swizzled K-major operand.
__host__ __device__ __forceinline__ uint32_t sw32_off(int n, int k) {
  return (n >> 3) * 256 + (n & 7) * 32 + ((((k >> 4) ^ (n >> 2)) & 1) << 4) + (k & 15);
}

// ------------------------------------------------------------ query prep --
// One warp per (request, head): lane i owns dims 16i..16i+15 of the latent
// query and lanes 0-3 also rope dims 16i..16i+15.  Writes the two E4M3 parts
// into the request's query image (rows n = part * 2NH + half * NH + head, the
// K index running over the half's 256 latent dims then its 32 rope dims) and
// the head's factor 2^-a.
template <int NH>
__global__ void __launch_bounds__(256) q8_prep_kernel(const Fp8PrepParams p) {
  using C = Cfg<NH>;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  // the decode kernel may launch now; it waits (griddepcontrol.wait) for this grid before reading
  griddep_launch_dependents();
  if (gw >= p.rows) return;
  const int b = gw / NH, h = gw % NH;
  const uint4* qn = reinterpret_cast<const uint4*>(p.q_nope + static_cast<size_t>(gw) * kLatent);
  const uint4* qr = reinterpret_cast<const uint4*>(p.q_rope + static_cast<size_t>(gw) * kRope);
  uint4 raw[2][2];
  raw[0][0] = qn[2 * lane];
  raw[0][1] = qn[2 * lane + 1];
  if (lane < 4) {
    raw[1][0] = qr[2 * lane];
    raw[1][1] = qr[2 * lane + 1];
  } else {
    raw[1][0] = raw[1][1] = make_uint4(0, 0, 0, 0);
  }
  float x[2][16];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(raw[c]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[c][2 * i] = __uint_as_float(w[i] << 16);
      x[c][2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[c][i]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  // a = 8 - e for amax = m 2^e, m in [0.5, 1): max |q 2^a| in [128, 256)
  int a = 0;
  if (amax > 0.f && amax <= 3.0e38f) {
    int e;
    frexpf(amax, &e);
    a = min(126, max(-126, 8 - e));
  }
  const float up = ldexpf(1.f, a);
  uint8_t* img = p.img + static_cast<size_t>(b) * C::kImg;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    if (c == 1 && lane >= 4) break;
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float u0 = x[c][2 * i] * up, u1 = x[c][2 * i + 1] * up;
      const uint32_t h2 = e4m3x2(u0, u1);
      const float2 hv = e4m3x2_value(h2);
      const uint32_t l2 = e4m3x2((u0 - hv.x) * 32.f, (u1 - hv.y) * 32.f);
      if (i & 1) {
        hi[i >> 1] |= h2 << 16;
        lo[i >> 1] |= l2 << 16;
      } else {
        hi[i >> 1] = h2;
        lo[i >> 1] = l2;
      }
    }
    int half, off_hi, off_lo;
    if (c == 0) {
      // latent dims 16 lane .. : half lane >> 4, K byte (16 lane) % 256 -> column (lane >> 3) & 1
      half = lane >> 4;
      const int k = (16 * lane) & 255;
      const int col = k >> 7;
      const int nh = half * NH + h, nl = 2 * NH + half * NH + h;
      off_hi = col * C::kR128 + sw128_off(nh, k & 127);
      off_lo = col * C::kR128 + sw128_off(nl, k & 127);
    } else {
      // rope dims 16 lane .. : half lane >> 1, K byte 16 (lane & 1) of the rope column
      half = lane >> 1;
      const int k = 16 * (lane & 1);
      const int nh = half * NH + h, nl = 2 * NH + half * NH + h;
      off_hi = 2 * C::kR128 + sw32_off(nh, k);
      off_lo = 2 * C::kR128 + sw32_off(nl, k);
    }
    *reinterpret_cast<uint4*>(img + off_hi) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(img + off_lo) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
  if (lane == 0) p.fac[gw] = ldexpf(1.f, -a);
}

// ------------------------------------------------------------ decode kernel --
template <int NH>
__global__ void __launch_bounds__(kThreads, 1)
    swab8_kernel(const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope,
                 const DecodeParams p, const Fp8Params p8) {
  using C = Cfg<NH>;
  constexpr int kHalf = C::kHalf;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return base + C::kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  int* last_armed = reinterpret_cast<int*>(smem + C::kOffLast);
  const WaitCtx wc{abort_flag, p.status};

  const int w = blockIdx.x;
  int it0, it1;
  plan_items(p, w, it0, it1);
  const int32_t* items = p.plan + p.items_off;
  const int nnz = __ldg(p.kv_indptr + p.batch);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kUnits; ++i) { mbar_init(bar(C::bFull + i), 1); mbar_init(bar(C::bEmpty + i), 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::bSFull + i), 1); mbar_init(bar(C::bSEmpty + i), 4);
      mbar_init(bar(C::bPFull + i), 4); mbar_init(bar(C::bPDone + i), 1);
      mbar_init(bar(C::bOBlk + i), 1);
    }
    mbar_init(bar(C::bQFull), 1); mbar_init(bar(C::bQEmpty), 1);
    mbar_init(bar(C::bOEmpty), 4);
    mbar_init(bar(C::bDrain), 2);
    for (int i = 0; i < C::kUnits; ++i) last_armed[i] = -1;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kPvWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  if (warp >= kProducerWarp0) {
    // ------------------------------------------------------ gather producers
    // Job j: token half th = j >> 2 of every tile, latent atom a = j & 3.
    // Lanes 0-7 gather the atom's 8 groups of 4 tokens (128-B rows); lanes
    // 8-11 gather rope groups 2a, 2a+1 of the half, from dim 512 (R0) and
    // from dim 544 (R1), 32-B rows.  Job 0 arms the unit's barrier with the
    // unit's bytes.  An out-of-range slot reads row 0 and sets
    // MLA_ERR_INDEX_OOB; the ragged tail repeats the last valid slot.
    const int job = warp - kProducerWarp0;
    const int th = job >> 2, a = job & 3;
    if (lane == 0 && job == 0) { tma_prefetch_desc(&tm_lat); tma_prefetch_desc(&tm_rope); }
    const bool active = lane < 12;
    const bool rope = lane >= 8;
    const int grp = rope ? 2 * a + ((lane - 8) & 1) : lane;       // group of 4 tokens within the half
    const int which = rope ? (lane - 8) >> 1 : 0;                 // R0 / R1
    const int tb = 32 * th + 4 * grp;                             // first token of the group in the tile
    const uint32_t dst_off = rope ? kRopeOff + which * kRopeAtom + (8 * th + grp) * 128
                                  : atom_pos(a) * kAtom + (8 * th + grp) * 512;
    const int x = rope ? kLatent + 32 * which : 128 * a;
    const CUtensorMap* map = rope ? &tm_rope : &tm_lat;
    const uint64_t pol = l2_policy_evict_first();
    uint32_t g = 0;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
      if (!item_ok(p, nnz, b, s, e)) {
        if (lane == 0 && job == 0) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
        continue;
      }
      const bool in_req = job != 0 || item_in_request(p, b, s, e);
      const int n = e - s;
      for (int t0 = 0; t0 < n && ok; t0 += T, ++g) {
        int v[4];
        bool oob = false;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          v[q] = __ldg(p.kv_indices + s + min(t0 + tb + q, n - 1));
          if (v[q] < 0 || static_cast<long long>(v[q]) >= p.num_slots) { oob = true; v[q] = 0; }
        }
        if (oob && !rope && a == 0) record_status(p.status, MLA_ERR_INDEX_OOB);   // jobs 0, 4 see every token
        const uint32_t slot = g % C::kUnits, use = g / C::kUnits;
        const uint32_t full = bar(C::bFull + slot);
        bool e_ok = true;
        if (lane == 0 && use > 0) e_ok = mbar_wait(bar(C::bEmpty + slot), (use - 1) & 1, wc);
        if (lane == 0 && e_ok && g >= static_cast<uint32_t>(kLead)) {
          const uint32_t gp = g - kLead;
          e_ok = mbar_wait(bar(C::bFull + gp % C::kUnits), (gp / C::kUnits) & 1, wc);
        }
        e_ok = __shfl_sync(0xffffffffu, e_ok, 0);
        if (!e_ok) { ok = false; break; }
        if (lane == 0 && job == 0) mbar_arrive_expect_tx(full, kUnit);
        __syncwarp();
        if (active)
          tma_gather4(base + C::kOffUnit + slot * kUnit + dst_off, map, x, v[0], v[1], v[2], v[3], full, pol);
        if (lane == 0 && job == 0) last_armed[slot] = static_cast<int>(use);
      }
      if (!in_req && lane == 0) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
    }
    // drain: every armed unit has landed before the CTA can exit
    named_bar_sync(kBarProd, 32 * kProducers);
    if (job == 0) {
      for (int i = lane; i < C::kUnits; i += 32) {
        const int uu = last_armed[i];
        if (uu >= 0) drain_wait(bar(C::bFull + i), uu & 1);
      }
    }
    __syncwarp();
  } else if (warp == kQkWarp) {
    // ------------------------------------------- QK issuer + query-image loader
    if (lane == 0) {
      griddep_wait();   // the query images come from the prep kernel
      const uint32_t qb = base + C::kOffQ;
      uint32_t g = 0, nitem = 0, us = 0, uph = 0;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
        if (!item_ok(p, nnz, b, s, e)) continue;
        const int nt = (e - s + T - 1) / T;
        if (nitem > 0 && !mbar_wait(bar(C::bQEmpty), (nitem - 1) & 1, wc)) break;
        mbar_arrive_expect_tx(bar(C::bQFull), C::kImg);
        bulk_load(qb, p8.img + static_cast<size_t>(b) * C::kImg, C::kImg, bar(C::bQFull));
        if (!mbar_wait(bar(C::bQFull), nitem & 1, wc)) break;
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t d_s = tmem + C::kTmS + (g & 1) * 4 * NH;
          if (g >= 2 && !mbar_wait(bar(C::bSEmpty + (g & 1)), ((g >> 1) - 1) & 1, wc)) { ok = false; break; }
          if (!mbar_wait(bar(C::bFull + us), uph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t ub = base + C::kOffUnit + us * kUnit;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            umma_ss_f8(d_s, sdesc(ub + (k >> 2) * 2 * kAtom + (k & 3) * 32, 16, 1024),
                       sdesc(qb + (k >> 2) * C::kR128 + (k & 3) * 32, 16, 1024), C::kIdescQK, k > 0 ? 1u : 0u);
          umma_ss_f8(d_s, sdesc(ub + kRopeOff, 16, 256, kLayoutSw32), sdesc(qb + 2 * C::kR128, 16, 256, kLayoutSw32),
                     C::kIdescQK, 1u);
          umma_commit(bar(C::bSFull + (g & 1)));
          if (j == nt - 1) umma_commit(bar(C::bQEmpty));
          if (++us == static_cast<uint32_t>(C::kUnits)) { us = 0; uph ^= 1; }
        }
        ++nitem;
      }
      umma_commit(bar(C::bDrain));
      drain_wait(bar(C::bDrain), 0);
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ PV issuer
    // A tile's PV once its [Phi; Plo]^T is written: O^T block mb (dims
    // 128mb..) += V^T (atom mb, MN-major) . P^T, two K-steps of 32 tokens;
    // then the unit is released.
    if (lane == 0) {
      uint32_t g = 0, nitem = 0, us = 0;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
        if (!item_ok(p, nnz, b, s, e)) continue;
        const int nt = (e - s + T - 1) / T;
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t buf = g & 1;
          if (!mbar_wait(bar(C::bPFull + buf), (g >> 1) & 1, wc)) { ok = false; break; }
          if (j == 0 && nitem > 0 && !mbar_wait(bar(C::bOEmpty), (nitem - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t ub = base + C::kOffUnit + us * kUnit;
          const uint32_t pb = base + C::kOffP + buf * C::kPBuf;
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
            for (int ks = 0; ks < 2; ++ks)
              umma_ss_f8(tmem + C::kTmO + mb * 2 * NH, sdesc(ub + atom_pos(mb) * kAtom + 4096 * ks, kAtom, 1024),
                         sdesc(pb + 32 * ks, 16, 1024), C::kIdescPV, (j == 0 && ks == 0) ? 0u : 1u);
            if (j == nt - 1 && (mb & 1)) umma_commit(bar(C::bOBlk + (mb >> 1)));
          }
          umma_commit(bar(C::bEmpty + us));
          us = (us + 1 == static_cast<uint32_t>(C::kUnits)) ? 0 : us + 1;
          umma_commit(bar(C::bPDone + buf));
        }
        ++nitem;
      }
      umma_commit(bar(C::bDrain));
      drain_wait(bar(C::bDrain), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- softmax + epilogue
    // As in the bf16 kernel: warps 0-1 hold the h0 partials of the tile's 64
    // tokens, warps 2-3 the h1 partials; each pair keeps half the heads and
    // hands the other half over through shared memory.  A partial is read as
    // hi + lo / 32 from its two column groups.
    const int pair = warp >> 1, wip = warp & 1;
    const int t = 32 * wip + lane;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float* X = reinterpret_cast<float*>(smem + C::kOffX);
    float* red = reinterpret_cast<float*>(smem + C::kOffRed);
    float* bc = reinterpret_cast<float*>(smem + C::kOffBc);
    int rk = 0;
    uint32_t g = 0, nitem = 0;
    bool aborted = false;
    float m_ref[kHalf], l_part[kHalf], fac[kHalf];
    auto wait = [&](uint32_t bb, uint32_t par) {
      if (aborted) return;
      bool r = true;
      if (lane == 0) r = mbar_wait(bb, par, wc);
      r = __shfl_sync(0xffffffffu, r, 0);
      if (!r) aborted = true;
    };
    griddep_wait();   // the per-head factors come from the prep kernel
    const float kv_scale = p8.kv_scale;

    for (int it = it0; it < it1; ++it) {
      const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
      const int part = items[4 * it + 3];
      if (!item_ok(p, nnz, b, s, e)) continue;
      // score factor of each own head: log2(e) sm_scale kv_scale 2^-a
#pragma unroll
      for (int k = 0; k < kHalf; ++k)
        fac[k] = p8.fac[static_cast<size_t>(b) * NH + pair * kHalf + k] * p.scale_log2 * kv_scale;
      const int n = e - s, nt = (n + T - 1) / T;
      for (int j = 0; j < nt; ++j, ++g) {
        const uint32_t buf = g & 1;
        wait(bar(C::bSFull + buf), (g >> 1) & 1);
        tc_fence_after();
        float ps[NH];
        if (!aborted) {
          uint32_t r[NH];
          const uint32_t ts = tmem + lane_off + C::kTmS + buf * 4 * NH + pair * NH;
          tmem_ld_cols<NH>(ts, r);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < NH; ++h) ps[h] = __uint_as_float(r[h]);
          tmem_ld_cols<NH>(ts + 2 * NH, r);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < NH; ++h) ps[h] = fmaf(__uint_as_float(r[h]), kLoWeight, ps[h]);
        } else {
#pragma unroll
          for (int h = 0; h < NH; ++h) ps[h] = 0.f;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(C::bSEmpty + buf));
        float own[kHalf];
#pragma unroll
        for (int k = 0; k < kHalf; ++k) {
          own[k] = pair ? ps[kHalf + k] : ps[k];
          X[(pair * kHalf + k) * T + t] = pair ? ps[k] : ps[kHalf + k];
        }
        named_bar_sync(kBarSm, 128);
        const bool valid = t < n - j * T;
        float sv[kHalf];
#pragma unroll
        for (int k = 0; k < kHalf; ++k)
          sv[k] = valid ? (own[k] + X[((1 - pair) * kHalf + k) * T + t]) * fac[k] : -INFINITY;
        if (j == 0) {
#pragma unroll
          for (int k = 0; k < kHalf; ++k) { m_ref[k] = sv[k]; l_part[k] = 0.f; }
          pair_reduce<kHalf, false>(m_ref, red, pair, wip, lane, rk);
          named_bar_sync(kBarVote, 128);
        } else {
          bool need = false;
#pragma unroll
          for (int k = 0; k < kHalf; ++k) need |= sv[k] > m_ref[k] + 8.f;
          need = named_bar_or(kBarVote, 128, need);
          if (need) {
            float mt[kHalf], alpha[kHalf];
#pragma unroll
            for (int k = 0; k < kHalf; ++k) mt[k] = sv[k];
            pair_reduce<kHalf, false>(mt, red, pair, wip, lane, rk);
#pragma unroll
            for (int k = 0; k < kHalf; ++k) {
              const float mn = fmaxf(m_ref[k], mt[k]);
              alpha[k] = ex2_approx(m_ref[k] - mn);
              m_ref[k] = mn;
              l_part[k] *= alpha[k];
            }
            if (wip == 0 && lane == 0) {
#pragma unroll
              for (int k = 0; k < kHalf; ++k) bc[pair * kHalf + k] = alpha[k];
            }
            named_bar_sync(kBarSm, 128);
            float alpha_all[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) alpha_all[h] = bc[h];
            wait(bar(C::bPDone + ((g - 1) & 1)), ((g - 1) >> 1) & 1);
            tc_fence_after();
            if (!aborted) {
#pragma unroll 1
              for (int c = 0; c < 8; ++c) {          // block c >> 1, hi (c even) or lo columns
                uint32_t o[NH];
                const uint32_t ta = tmem + lane_off + C::kTmO + c * NH;
                tmem_ld_cols<NH>(ta, o);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < NH; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha_all[h]);
                tmem_st_cols<NH>(ta, o);
              }
              tmem_wait_st();
            }
          }
        }
        // weights: hi + lo / 32 in E4M3, summed as the MMA will see them
        uint32_t phi[kHalf / 2], plo[kHalf / 2];
#pragma unroll
        for (int k = 0; k < kHalf; k += 2) {
          const float p0 = ex2_approx(sv[k] - m_ref[k]), p1 = ex2_approx(sv[k + 1] - m_ref[k + 1]);
          const uint32_t h2 = e4m3x2(p0, p1);
          const float2 hv = e4m3x2_value(h2);
          const uint32_t l2 = e4m3x2((p0 - hv.x) * 32.f, (p1 - hv.y) * 32.f);
          const float2 lv = e4m3x2_value(l2);
          l_part[k] += fmaf(lv.x, kLoWeight, hv.x);
          l_part[k + 1] += fmaf(lv.y, kLoWeight, hv.y);
          phi[k >> 1] = h2;
          plo[k >> 1] = l2;
        }
        if (g >= 2) wait(bar(C::bPDone + buf), ((g >> 1) - 1) & 1);
        if (!aborted) {
          // [Phi; Plo]^T[buf]: K-major, 128-B swizzle; row = head (hi) or NH + head (lo), byte = token
          uint8_t* pb = smem + C::kOffP + buf * C::kPBuf;
#pragma unroll
          for (int k = 0; k < kHalf; k += 2) {
            const int h = pair * kHalf + k;
            pb[sw128_off(h, t)] = static_cast<uint8_t>(phi[k >> 1]);
            pb[sw128_off(h + 1, t)] = static_cast<uint8_t>(phi[k >> 1] >> 8);
            pb[sw128_off(NH + h, t)] = static_cast<uint8_t>(plo[k >> 1]);
            pb[sw128_off(NH + h + 1, t)] = static_cast<uint8_t>(plo[k >> 1] >> 8);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(C::bPFull + buf));
      }
      // ------------------------------------------------------------ epilogue
      const bool tid0 = threadIdx.x == 0;
      const bool to_out = part < 0;
      const bool part_ok = part < p.max_partials;   // a device-only plan naming a partial past the workspace
      if (!part_ok && tid0) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
      float l_tot[kHalf];
#pragma unroll
      for (int k = 0; k < kHalf; ++k) l_tot[k] = l_part[k];
      pair_reduce<kHalf, true>(l_tot, red, pair, wip, lane, rk);
      if (wip == 0 && lane == 0) {
#pragma unroll
        for (int k = 0; k < kHalf; k += 4)
          *reinterpret_cast<float4*>(bc + pair * kHalf + k) = make_float4(
              __frcp_rn(l_tot[k]), __frcp_rn(l_tot[k + 1]), __frcp_rn(l_tot[k + 2]), __frcp_rn(l_tot[k + 3]));
      }
      {
        float my_lse = 0.f;
#pragma unroll
        for (int k = 0; k < kHalf; ++k)
          if (lane == k) my_lse = (m_ref[k] + __log2f(l_tot[k])) * 0.69314718055994531f;
        if (!aborted && part_ok && wip == 0 && lane < kHalf) {
          const int h = pair * kHalf + lane;
          if (to_out) { if (p.lse) p.lse[static_cast<size_t>(b) * p.heads + h] = my_lse; }
          else p.part_lse[static_cast<size_t>(part) * p.heads + h] = my_lse;
        }
      }
      named_bar_sync(kBarSm, 128);
      float inv_l[NH];   // 1/l and the cache scale
#pragma unroll
      for (int h = 0; h < NH; ++h) inv_l[h] = bc[h] * kv_scale;
      const bool st_bf16 = to_out && p.out_bf16;
      const int esz = st_bf16 ? 2 : 4;
      uint8_t* dst = to_out ? reinterpret_cast<uint8_t*>(p.out) + static_cast<size_t>(b) * p.heads * kLatent * esz
                            : reinterpret_cast<uint8_t*>(p.part_o + static_cast<size_t>(part) * p.heads * kLatent);
      uint8_t* wst = smem + C::kOffX + warp * NH * 32 * 4;
      const int lg = st_bf16 ? 2 : 3;
#pragma unroll 1
      for (int mb = 0; mb < 4; ++mb) {
        if ((mb & 1) == 0) {
          wait(bar(C::bOBlk + (mb >> 1)), nitem & 1);
          tc_fence_after();
        }
        float v[NH];
        if (!aborted) {
          uint32_t o[NH];
          const uint32_t ta = tmem + lane_off + C::kTmO + mb * 2 * NH;
          tmem_ld_cols<NH>(ta, o);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < NH; ++h) v[h] = __uint_as_float(o[h]);
          tmem_ld_cols<NH>(ta + NH, o);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < NH; ++h) v[h] = fmaf(__uint_as_float(o[h]), kLoWeight, v[h]) * inv_l[h];
        } else {
#pragma unroll
          for (int h = 0; h < NH; ++h) v[h] = 0.f;
        }
        if (mb == 3) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0 && !aborted) mbar_arrive(bar(C::bOEmpty));
        }
        if (st_bf16) {
#pragma unroll
          for (int h = 0; h < NH; ++h) reinterpret_cast<__nv_bfloat16*>(wst)[h * 32 + lane] = __float2bfloat16_rn(v[h]);
        } else {
#pragma unroll
          for (int h = 0; h < NH; ++h) reinterpret_cast<float*>(wst)[h * 32 + lane] = v[h];
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < NH * 8 / 32; ++k) {
          const int c = lane + 32 * k;
          if (c < (NH << lg) && !aborted && part_ok) {
            const int h = c >> lg, cc = c & ((1 << lg) - 1);
            const uint4 val = *reinterpret_cast<const uint4*>(wst + (h * 32) * esz + 16 * cc);
            *reinterpret_cast<uint4*>(dst + (static_cast<size_t>(h) * kLatent + 128 * mb + 32 * warp) * esz + 16 * cc) =
                val;
          }
        }
        __syncwarp();
      }
      named_bar_sync(kBarSm, 128);   // the staging rows double as the next tile's exchange buffer
      ++nitem;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kPvWarp) tmem_dealloc(tmem, C::kTmemCols);
}

// ------------------------------------------------------------ FP8 append --
// Request r's new bf16 row goes to slot slots[r] as E4M3 codes of value /
// kv_scale (IEEE float32 division, then round to nearest even, saturating at
// 448).  One thread per 16 output bytes, eight rows per 288-thread block.
constexpr int kAppendPieces = kRow / 16;   // 36
constexpr int kAppendRows = 8;

__global__ void __launch_bounds__(kAppendPieces * kAppendRows) append_fp8_kernel(const AppendFp8Params p) {
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
  const uint4* src = reinterpret_cast<const uint4*>(p.src + static_cast<size_t>(r) * kRow) + 2 * piece;
  const uint4 w0 = __ldg(src), w1 = __ldg(src + 1);
  const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a = __fdiv_rn(__uint_as_float(w[i] << 16), p.kv_scale);
    const float b = __fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), p.kv_scale);
    const uint32_t c = e4m3x2(a, b);
    if (i & 1) out[i >> 1] |= c << 16;
    else out[i >> 1] = c;
  }
  *reinterpret_cast<uint4*>(p.kv_cache + slot * kRow + 16 * piece) = make_uint4(out[0], out[1], out[2], out[3]);
}

template <int NH>
int launch(const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const DecodeParams& p, const Fp8Params& p8,
           const Fp8PrepParams& pp, int grid, cudaStream_t stream) {
  using C = Cfg<NH>;
  if (!set_smem_limit(reinterpret_cast<const void*>(&swab8_kernel<NH>), C::kSmemBytes)) return MLA_ERR_CUDA;
  const int warps = pp.rows;
  // a plain launch (full stream order): the decode kernel below, its
  // programmatic dependent, starts gathering cache rows before it waits, which
  // is safe only because everything before the prep kernel has finished
  q8_prep_kernel<NH><<<(warps + 7) / 8, 256, 0, stream>>>(pp);
  if (cudaPeekAtLastError() != cudaSuccess) return MLA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, swab8_kernel<NH>, tm_lat, tm_rope, p, p8) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // namespace swab8

int launch_swab8(int heads, const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const DecodeParams& p,
                 const Fp8Params& p8, const Fp8PrepParams& pp, int grid, cudaStream_t stream) {
  if (heads == 16) return swab8::launch<16>(tm_lat, tm_rope, p, p8, pp, grid, stream);
  if (heads == 32) return swab8::launch<32>(tm_lat, tm_rope, p, p8, pp, grid, stream);
  return MLA_ERR_UNSUPPORTED;
}

size_t fp8_image_bytes(int heads) { return static_cast<size_t>(4) * heads * 288; }

int launch_append_fp8(const AppendFp8Params& p, cudaStream_t stream) {
  if (p.rows <= 0) return MLA_OK;
  const int blocks = (p.rows + swab8::kAppendRows - 1) / swab8::kAppendRows;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(swab8::kAppendPieces * swab8::kAppendRows, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, swab8::append_fp8_kernel, p) != cudaSuccess) return MLA_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace mla
