// Absorbed MLA decode for few heads (H = 16 or 32) on sm_103a.
//
// With only 16 or 32 query heads the tensor core's M side cannot be the
// heads, so both products run "swapped": tokens (or latent dims) on M, heads
// on N.  A tcgen05.mma costs about the same ~50 cycles whatever its M (64 or
// 128) and its N (16..64), so the kernel is built to issue as few as possible:
//
//   QK, folded: the 576 score dims are split into two halves,
//       h0 = latent atoms 0-3 + rope dims 0-31,  h1 = latent atoms 4-7 + rope dims 32-63,
//     and the two halves of a 64-token tile are stacked on M:
//       D[128 x 2H] = [K_h0; K_h1] (128 rows) . [Q_h0; Q_h1]^T (2H rows), K = 288
//     Rows 0-63 x cols [0,H) hold the h0 partial score, rows 64-127 x cols
//     [H,2H) the h1 partial (the two off-diagonal blocks are never read), so
//     a tile takes 18 MMAs instead of 36.  S = partial_h0 + partial_h1.
//   PV: O^T[128 dims x H] += V^T[128 dims x 64 tok] . P^T[64 tok x H]   (4 blocks of M = 128 dims,
//                                                                          A read MN-major from the same atoms)
//
// The rows of a request are gathered from the page-size-1 cache with TMA
// gather4 (four slots per instruction) into 128-byte-swizzled "atoms" of 64
// tokens x 64 dims (8 KB).  A tile lands in three ring units: latent unit A
// holds atoms {0, 4, 1, 5}, unit B atoms {2, 6, 3, 7} (so atom c+4 follows
// atom c and one 128-row descriptor covers both halves), and the rope unit
// holds rope dims 0-31 then 32-63 as two atoms of 64 tokens x 32 dims (64-byte
// rows, 64-byte swizzle), so one 128-row descriptor covers the rope of both
// halves too and no byte past the row is gathered.  Each latent byte is read
// by the tensor core twice -- in the key (score over 576) and as the value
// (the latent reused as V) -- and its unit is released after its PVs, so
// every cache byte crosses HBM once.
// ("实现差距：MLA 与 DeepSeek V3", section 2.4: dual-path score, FA2-style
// online softmax, kv_c reused as the value; "Attention backends", paragraph
// "MLA": 576 wide for k and 512 for v, one shared vector per token.)
//
// Warp roles (one CTA per SM, persistent over the plan's work items):
//   warps 0-3   softmax / epilogue / merge (TMEM lane quadrants 0-3)
//   warp 4      QK issuer and query loader (one thread, blocking waits)
//   warp 5      TMEM allocator and PV issuer (one thread, blocking waits)
//   warps 6-15  gather producers, one gather job (16 gather4) of every tile
//               each; a producer reads its tile's slot numbers itself
//
// Softmax: warps 0-1 read the h0 partials of tokens 0-63 (lanes 0-63), warps
// 2-3 the h1 partials (lanes 64-127); each pair keeps half the heads and
// hands the other half to its partner through shared memory, so each of the
// 128 threads finishes one token for H/2 heads.  Scores are in log2 units;
// each head keeps a reference maximum m_ref that only moves when a tile
// exceeds it by more than 8 (a vote per tile); then O and the running sums
// are rescaled once.  So P = 2^(s - m_ref) <= 256 always fits bf16.
//
// Epilogue: O^T is scaled by 1/l, staged in shared memory and written with
// 16-byte stores (a warp writes 512 contiguous bytes), to out/lse for a
// request the plan left whole, else as an fp32 partial state for the merge
// kernel, which is launched as a programmatic dependent of this kernel.
#include "mla_device.cuh"
#include "mla_launch.h"

namespace mla {
namespace swab {

constexpr int T = 64;                      // tokens per tile
constexpr int kQkWarp = 4, kPvWarp = 5, kProducerWarp0 = 6;
constexpr int kProducers = 10;             // latent atoms 0-7, rope dims 0-31, rope dims 32-63
constexpr int kThreads = 32 * (kProducerWarp0 + kProducers);
constexpr int kAtom = T * 128;             // 8 KB: 64 tokens x 64 dims
constexpr int kUnit = 4 * kAtom;           // latent unit: atoms {c, c+4, c+1, c+5}
constexpr int kRopeAtom = T * 64;          // 4 KB: 64 tokens x 32 rope dims (64-byte swizzle)
constexpr int kRopeUnit = 2 * kRopeAtom;   // rope dims 0-31, then 32-63
constexpr int kRopeUnits = 2;
#ifndef MLA_SWAB_LEAD_UNITS
#define MLA_SWAB_LEAD_UNITS 4
#endif
// Pacing: a producer issues latent unit s only once unit s - kLeadUnits has
// landed (and rope unit g once rope unit g - kLeadRope has), which bounds the
// bytes in flight per SM; more would only lengthen the memory queues.
constexpr int kLeadUnits = MLA_SWAB_LEAD_UNITS;
constexpr int kLeadRope = (kLeadUnits + 1) / 2;
static_assert(kLeadRope <= kRopeUnits, "a rope slot's phase must not be lapped while it is waited on");
constexpr int kBarSm = 1, kBarVote = 2, kBarPair0 = 3, kBarProd = 5;   // named barriers

template <int NH>
struct Cfg {
  static constexpr int kHalf = NH / 2;
  static constexpr int kLatUnits = (NH == 16) ? 5 : 4;   // 2.5 or 2 tiles of latent
  static_assert(kLeadUnits <= kLatUnits, "a latent slot's phase must not be lapped while it is waited on");
  static constexpr int kQPair = 2 * NH * 128;            // two Q atoms of NH rows
  static constexpr int kQBytes = 5 * kQPair;             // 4 latent pairs + the rope pair
  static constexpr int kPBuf = NH * 128;                 // P^T: NH heads x 64 tokens bf16
  static constexpr int kXBytes = 2 * kHalf * T * 4;      // partial-score exchange, both directions
  static constexpr int kStage = NH * 128 * 4;            // epilogue staging: 4 warps x [NH][32] fp32
  static constexpr int kOffLat = 0;
  static constexpr int kOffRope = kOffLat + kLatUnits * kUnit;
  static constexpr int kOffQ = kOffRope + kRopeUnits * kRopeUnit;
  static constexpr int kOffP = kOffQ + kQBytes;
  static constexpr int kOffX = kOffP + 2 * kPBuf;
  static constexpr int kOffRed = kOffX + kStage;         // [2 bufs][2 pairs][2 warps][kHalf] floats
  static constexpr int kOffBc = kOffRed + 8 * kHalf * 4; // [NH] floats: alpha, then 1/l
  // barrier indices
  static constexpr int bLatFull = 0;
  static constexpr int bLatEmpty = bLatFull + kLatUnits;
  static constexpr int bRopeFull = bLatEmpty + kLatUnits;
  static constexpr int bRopeEmpty = bRopeFull + kRopeUnits;
  static constexpr int bQFull = bRopeEmpty + kRopeUnits;
  static constexpr int bQEmpty = bQFull + 1;
  static constexpr int bSFull = bQEmpty + 1;             // [2] QK(g) is in S buffer g&1
  static constexpr int bSEmpty = bSFull + 2;             // [2] the softmax has read it
  static constexpr int bPFull = bSEmpty + 2;             // [2] P(g) is in P buffer g&1
  static constexpr int bPDone = bPFull + 2;              // [2] PV(g) has completed
  static constexpr int bOBlk = bPDone + 2;               // [4] an item's last PV of O^T block mb is done
  static constexpr int bOEmpty = bOBlk + 4;
  static constexpr int bDrain = bOEmpty + 1;             // both issuers' final commits
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kOffBar = kOffBc + NH * 4;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem slot, abort flag, merge decision
  static constexpr int kOffLast = kOffMisc + 32;            // [kLatUnits + kRopeUnits] last armed use
  static constexpr int kSmemBytes = kOffLast + 4 * (kLatUnits + kRopeUnits) + 1024;   // + alignment slack
  static constexpr int kTmemCols = 8 * NH;                  // S: 2 x 2NH, O^T: 4 x NH
  static constexpr int kTmS = 0;
  static constexpr int kTmO = 4 * NH;
  static constexpr uint32_t kIdescQK = idesc_bf16(128, 2 * NH, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16(128, NH, true, false);
  static_assert(kStage >= kXBytes, "the exchange and the epilogue staging share a region");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kPBuf % 1024 == 0 && kQPair % 1024 == 0,
                "atoms must be 1024-byte aligned");
  static_assert(kOffBar % 8 == 0, "alignment");
};

// Items every role processes: a request in range and a token range inside
// kv_indices (so no access can leave the arrays).  Whether the range also
// lies inside its own request is checked off the critical path by one
// producer (item_in_request), which only records MLA_ERR_PLAN_MISMATCH.
__device__ __forceinline__ bool item_ok(const DecodeParams& p, int nnz, int b, int s, int e) {
  return b >= 0 && b < p.batch && 0 <= s && s < e && e <= nnz;
}
__device__ __forceinline__ bool item_in_request(const DecodeParams& p, int b, int s, int e) {
  const int lo = __ldg(p.kv_indptr + b), hi = __ldg(p.kv_indptr + b + 1);
  return lo <= s && e <= hi;
}

// Bounded wait that ignores the abort flag (used to drain in-flight copies).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > MLA_WAIT_LIMIT_NS) return;
  }
}

// Max (or sum) over the 64 threads of a warp pair -- the two warps that hold
// the same heads -- of v[i] for every i; both warps get the result.  `red` is
// [2 bufs][2 pairs][2 warps][K]; `k` alternates the buffer.
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
  static_assert(N % 16 == 0, "16-column loads");
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

// kMQ: several query tokens per request (q_len > 1), each row with its own
// causal limit; the single-query instantiation carries none of it.
template <int NH, bool kMQ>
__global__ void __launch_bounds__(kThreads, 1)
    swab_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_kr,
                const __grid_constant__ CUtensorMap tm_qn, const __grid_constant__ CUtensorMap tm_qr,
                const DecodeParams p) {
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
  int* last_armed = reinterpret_cast<int*>(smem + C::kOffLast);   // per ring slot: last armed use
  const WaitCtx wc{abort_flag, p.status};
#ifdef MLA_TRACE
  if (threadIdx.x == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    MLA_TRACE_RAW(15, 0, static_cast<long long>(globaltimer()));
    MLA_TRACE_RAW(15, 2, static_cast<long long>(smid));
    MLA_TRACE_RAW(15, 3, clock64());
  }
#endif

  const int w = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kLatUnits; ++i) { mbar_init(bar(C::bLatFull + i), 1); mbar_init(bar(C::bLatEmpty + i), 1); }
    for (int i = 0; i < kRopeUnits; ++i) { mbar_init(bar(C::bRopeFull + i), 1); mbar_init(bar(C::bRopeEmpty + i), 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::bSFull + i), 1); mbar_init(bar(C::bSEmpty + i), 4);
      mbar_init(bar(C::bPFull + i), 4); mbar_init(bar(C::bPDone + i), 1);
    }
    mbar_init(bar(C::bQFull), 1); mbar_init(bar(C::bQEmpty), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(C::bOBlk + i), 1);
    mbar_init(bar(C::bOEmpty), 4);
    mbar_init(bar(C::bDrain), 2);
    for (int i = 0; i < C::kLatUnits + kRopeUnits; ++i) last_armed[i] = -1;
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
  // launched as a programmatic dependent of the previous kernel in the
  // stream: everything above overlapped its tail; its results (the plan,
  // indices, query, cache rows) are read only after it has finished
  griddep_wait();
  int it0, it1;
  plan_items(p, w, it0, it1);
  const int32_t* items = p.plan + p.items_off;
  const int nnz = __ldg(p.kv_indptr + p.batch);
  if (threadIdx.x == 0) MLA_TRACE_RAW(15, 5, clock64());
  // the merge kernel may be launched now: it waits for this grid to finish
  griddep_launch_dependents();

  if (warp >= kProducerWarp0) {
    // ------------------------------------------------------ gather producers
    // A warp completes one gather4 only every ~70-110 cycles, so a tile's
    // landing time is set by how many gathers one warp issues for it: each
    // producer owns one of the tile's ten gather jobs (16 gather4 each).
    // Job k < 8 is latent atom k (unit (k >> 1) & 1, position 2(k & 1) + (k >> 2));
    // jobs 8 and 9 rope dims 0-31 and 32-63 (row dims 512..543, 544..575).
    // Jobs 0, 2 and 8 arm their unit's full barrier with the unit's bytes.
    // Slot numbers come straight from kv_indices (lane l < 16 loads tokens
    // 4l..4l+3, issued before the wait for ring space so the load overlaps
    // it); an out-of-range slot reads row 0 and sets MLA_ERR_INDEX_OOB, and
    // the ragged tail repeats the last valid slot (its scores are masked).
    const int job = warp - kProducerWarp0;
    if (lane == 0 && job == 0) tma_prefetch_desc(&tm_kv);
    if (lane == 0 && job == 8) tma_prefetch_desc(&tm_kr);
    const bool rope = job >= 8;
    const int u = (job >> 1) & 1;
    const int x = rope ? kLatent + 32 * (job - 8) : 64 * job;
    const uint32_t pos_off = rope ? (job - 8) * kRopeAtom : ((job & 1) * 2 + (job >> 2)) * kAtom;
    const CUtensorMap* tmap = rope ? &tm_kr : &tm_kv;
    const uint32_t row_bytes = rope ? 64u : 128u;            // per gathered row
    const bool arms = rope ? job == 8 : (job == 0 || job == 2);
    const uint32_t arm_bytes = rope ? kRopeUnit : kUnit;
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
          v[q] = __ldg(p.kv_indices + s + min(t0 + 4 * (lane & 15) + q, n - 1));
          if (v[q] < 0 || static_cast<long long>(v[q]) >= p.num_slots) { oob = true; v[q] = 0; }
        }
        if (oob && job == 0) record_status(p.status, MLA_ERR_INDEX_OOB);
        if (lane == 0 && job < 4) MLA_TRACE_EVENT(job == 0 ? 0 : 8 + job, g);
        uint32_t slot, use, addr, full, empty;
        int last_idx;
        if (rope) {
          slot = g % kRopeUnits;
          use = g / kRopeUnits;
          addr = base + C::kOffRope + slot * kRopeUnit;
          full = bar(C::bRopeFull + slot);
          empty = bar(C::bRopeEmpty + slot);
          last_idx = C::kLatUnits + slot;
        } else {
          const uint32_t seq = 2 * g + u;
          slot = seq % C::kLatUnits;
          use = seq / C::kLatUnits;
          addr = base + C::kOffLat + slot * kUnit;
          full = bar(C::bLatFull + slot);
          empty = bar(C::bLatEmpty + slot);
          last_idx = slot;
        }
        bool e_ok = true;
        if (lane == 0 && use > 0) e_ok = mbar_wait(empty, (use - 1) & 1, wc);
        if (lane == 0 && e_ok) {
          if (rope) {
            if (g >= static_cast<uint32_t>(kLeadRope)) {
              const uint32_t gp = g - kLeadRope;
              e_ok = mbar_wait(bar(C::bRopeFull + gp % kRopeUnits), (gp / kRopeUnits) & 1, wc);
            }
          } else if (2 * g + u >= static_cast<uint32_t>(kLeadUnits)) {
            const uint32_t sp = 2 * g + u - kLeadUnits;
            e_ok = mbar_wait(bar(C::bLatFull + sp % C::kLatUnits), (sp / C::kLatUnits) & 1, wc);
          }
        }
        e_ok = __shfl_sync(0xffffffffu, e_ok, 0);
        if (!e_ok) { ok = false; break; }
        if (lane == 0 && arms) mbar_arrive_expect_tx(full, arm_bytes);
        __syncwarp();
        if (lane < 16) tma_gather4(addr + pos_off + lane * 4 * row_bytes, tmap, x, v[0], v[1], v[2], v[3], full, pol);
        if (lane == 0 && arms) atomicMax(last_armed + last_idx, static_cast<int>(use));
        if (lane == 0 && job == 0) MLA_TRACE_EVENT(1, g);
      }
      if (!in_req && lane == 0) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
    }
    // drain: every copy armed by any producer has landed before the CTA can
    // exit (slots are shared between producer warps, so use the latest use)
    named_bar_sync(kBarProd, 32 * kProducers);
    if (job == 0) {
      for (int i = lane; i < C::kLatUnits + kRopeUnits; i += 32) {
        const int uu = last_armed[i];
        const int bfull = i < C::kLatUnits ? C::bLatFull + i : C::bRopeFull + (i - C::kLatUnits);
        if (uu >= 0) drain_wait(bar(bfull), uu & 1);
      }
    }
    __syncwarp();
  } else if (warp == kQkWarp) {
    // ----------------------------------------------- QK issuer + query loader
    // One thread that blocks on its barriers.  Per item it loads the query
    // (four latent atom pairs {c, c+4} and the rope pair) once the previous
    // item's last QK has read the old one; per tile it scores units A, B and
    // the rope unit as they land: 8 + 8 + 2 MMAs into S buffer g&1.
    if (lane == 0) {
      tma_prefetch_desc(&tm_qn);
      tma_prefetch_desc(&tm_qr);
      const uint64_t dq = sdesc(base + C::kOffQ, 16, 1024);      // Q pair 0 (B of QK)
      const uint64_t dk = sdesc(base + C::kOffLat, 16, 1024);    // latent unit slot 0 (A of QK)
      const uint64_t dr = sdesc(base + C::kOffRope, 16, 512, kLayoutSw64);   // rope unit slot 0 (A of QK)
      auto D = [](uint64_t d, uint32_t byte_off) -> uint64_t { return d + (byte_off >> 4); };
      const uint32_t qbase = base + C::kOffQ;
      uint32_t g = 0, nitem = 0, ls = 0, lph = 0, rs = 0, rph = 0;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
        if (!item_ok(p, nnz, b, s, e)) continue;
        const int nt = (e - s + T - 1) / T;
        if (nitem > 0 && !mbar_wait(bar(C::bQEmpty), (nitem - 1) & 1, wc)) break;
        mbar_arrive_expect_tx(bar(C::bQFull), C::kQBytes);
        for (int c = 0; c < 4; ++c) {
          tma_load_2d(qbase + c * C::kQPair, &tm_qn, 64 * c, b * p.heads, bar(C::bQFull));
          tma_load_2d(qbase + c * C::kQPair + NH * 128, &tm_qn, 64 * (c + 4), b * p.heads, bar(C::bQFull));
        }
        tma_load_2d(qbase + 4 * C::kQPair, &tm_qr, 0, b * p.heads, bar(C::bQFull));
        tma_load_2d(qbase + 4 * C::kQPair + NH * 128, &tm_qr, 32, b * p.heads, bar(C::bQFull));
        if (nitem < 8) MLA_TRACE_RAW(14, 2 * nitem, clock64());
        if (!mbar_wait(bar(C::bQFull), nitem & 1, wc)) break;
        if (nitem < 8) MLA_TRACE_RAW(14, 2 * nitem + 1, clock64());
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t d_s = tmem + C::kTmS + (g & 1) * 2 * NH;
          if (g >= 2 && !mbar_wait(bar(C::bSEmpty + (g & 1)), ((g >> 1) - 1) & 1, wc)) { ok = false; break; }
          MLA_TRACE_EVENT(2, g);
#pragma unroll 1
          for (int uu = 0; uu < 2 && ok; ++uu) {
            if (!mbar_wait(bar(C::bLatFull + ls), lph, wc)) { ok = false; break; }
            tc_fence_after();
            const uint64_t ak = D(dk, ls * kUnit);
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
              const uint64_t bq = D(dq, (2 * uu + pr) * C::kQPair);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_ss(d_s, D(ak, pr * 2 * kAtom + 32 * kk), D(bq, 32 * kk), C::kIdescQK,
                        (uu | pr | kk) != 0 ? 1u : 0u);
            }
            if (++ls == static_cast<uint32_t>(C::kLatUnits)) { ls = 0; lph ^= 1; }
          }
          if (!ok || !mbar_wait(bar(C::bRopeFull + rs), rph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ar = D(dr, rs * kRopeUnit);
          const uint64_t bq = D(dq, 4 * C::kQPair);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) umma_ss(d_s, D(ar, 32 * kk), D(bq, 32 * kk), C::kIdescQK, 1u);
          umma_commit(bar(C::bRopeEmpty + rs));
          if (++rs == static_cast<uint32_t>(kRopeUnits)) { rs = 0; rph ^= 1; }
          umma_commit(bar(C::bSFull + (g & 1)));
          if (j == nt - 1) umma_commit(bar(C::bQEmpty));
          MLA_TRACE_EVENT(3, g);
        }
        ++nitem;
      }
      umma_commit(bar(C::bDrain));
      drain_wait(bar(C::bDrain), 0);
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ PV issuer
    // Issues a tile's PV once its P^T is written: the two 128-dim blocks of
    // unit A (dims 0-127 = atoms 0,1 and dims 256-383 = atoms 4,5), then
    // unit A is released; the same for unit B (dims 128-255, 384-511).
    if (lane == 0) {
      const uint64_t dv = sdesc(base + C::kOffLat, 2 * kAtom, 1024);   // A of PV, MN-major: atoms 2 apart
      const uint64_t dp = sdesc(base + C::kOffP, 16, 1024);            // P^T buffer 0 (B of PV)
      auto D = [](uint64_t d, uint32_t byte_off) -> uint64_t { return d + (byte_off >> 4); };
      uint32_t g = 0, nitem = 0, ls = 0;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
        if (!item_ok(p, nnz, b, s, e)) continue;
        const int nt = (e - s + T - 1) / T;
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t buf = g & 1;
          if (!mbar_wait(bar(C::bPFull + buf), (g >> 1) & 1, wc)) { ok = false; break; }
          if (j == nt - 1 && nitem < 8) MLA_TRACE_RAW(12, 8 * nitem + 4, clock64());
          if (j == 0 && nitem > 0 && !mbar_wait(bar(C::bOEmpty), (nitem - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          MLA_TRACE_EVENT(4, g);
          const uint64_t bp = D(dp, buf * C::kPBuf);
#pragma unroll
          for (int uu = 0; uu < 2; ++uu) {
            const uint64_t au = D(dv, ls * kUnit);
#pragma unroll
            for (int hi = 0; hi < 2; ++hi) {
              const int mb = uu + 2 * hi;            // 128-dim block
              const uint64_t av = D(au, hi * kAtom);
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                umma_ss(tmem + C::kTmO + mb * NH, D(av, ks * 2048), D(bp, ks * 32), C::kIdescPV,
                        (j == 0 && ks == 0) ? 0u : 1u);
              if (j == nt - 1) umma_commit(bar(C::bOBlk + mb));   // the epilogue streams blocks as they finish
              if (j == nt - 1 && nitem < 8) MLA_TRACE_RAW(12, 8 * nitem + mb, clock64());
            }
            umma_commit(bar(C::bLatEmpty + ls));
            ls = (ls + 1 == static_cast<uint32_t>(C::kLatUnits)) ? 0 : ls + 1;
          }
          umma_commit(bar(C::bPDone + buf));
          MLA_TRACE_EVENT(5, g);
        }
        ++nitem;
      }
      umma_commit(bar(C::bDrain));
      drain_wait(bar(C::bDrain), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- softmax + epilogue
    const int pair = warp >> 1, wip = warp & 1;
    const int t = 32 * wip + lane;                        // token of the tile
    const int tid = threadIdx.x;                          // 0..127
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float* X = reinterpret_cast<float*>(smem + C::kOffX);
    float* red = reinterpret_cast<float*>(smem + C::kOffRed);
    float* bc = reinterpret_cast<float*>(smem + C::kOffBc);
    int rk = 0;
    uint32_t g = 0, nitem = 0;
    bool aborted = false;
    float m_ref[kHalf], l_part[kHalf];
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
      if (!item_ok(p, nnz, b, s, e)) continue;
      const int n = e - s, nt = (n + T - 1) / T;
      // multi-query: head row h is query i = h / (NH / q_len) of its request.
      // A chain of drafts sees the first L - q_len + 1 + i rows of the
      // request's context, i.e. the item's first mq_base + i tokens; a tree
      // sees the item's tokens before mq_d0 (the first draft) and, among the
      // drafts, the ancestors of draft i and draft i itself
      constexpr bool mq = kMQ;
      int mq_base = n, mq_heads = NH, mq_d0 = 0x3FFFFFFF;
      const bool tree = kMQ && p.tree_masks != nullptr;
      if (mq) {
        const int lo = __ldg(p.kv_indptr + b), hi = __ldg(p.kv_indptr + b + 1);
        mq_heads = NH / p.q_len;
        if (tree) mq_d0 = (hi - lo) - p.q_len - (s - lo);
        else mq_base = (hi - lo) - p.q_len + 1 - (s - lo);
      }
      const unsigned long long* anc_b = tree ? p.tree_masks + static_cast<size_t>(b) * p.q_len : nullptr;
      for (int j = 0; j < nt; ++j, ++g) {
        const uint32_t buf = g & 1;
        wait(bar(C::bSFull + buf), (g >> 1) & 1);
        if (tid == 0) MLA_TRACE_EVENT(6, g);
        tc_fence_after();
        uint32_t r[NH];
        if (!aborted) {
          tmem_ld_cols<NH>(tmem + lane_off + C::kTmS + buf * 2 * NH + pair * NH, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int h = 0; h < NH; ++h) r[h] = 0;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(C::bSEmpty + buf));
        // hand the partner pair the partials of its heads, take ours
        float own[kHalf];
#pragma unroll
        for (int k = 0; k < kHalf; ++k) {
          own[k] = __uint_as_float(pair ? r[kHalf + k] : r[k]);
          X[(pair * kHalf + k) * T + t] = __uint_as_float(pair ? r[k] : r[kHalf + k]);
        }
        named_bar_sync(kBarSm, 128);
        float sv[kHalf];
        const int kd = j * T + t - mq_d0;       // this token's draft index (tree), < 0 for the shared context
#pragma unroll
        for (int k = 0; k < kHalf; ++k) {
          const int lim = mq ? max(0, min(n, mq_base + (pair * kHalf + k) / mq_heads)) : n;
          bool ok = t < lim - j * T;
          if (kMQ && kd >= 0)                     // only a tree's draft tokens: an ancestor of this row's query?
            ok = ok && kd < 64 && ((__ldg(anc_b + (pair * kHalf + k) / mq_heads) >> kd) & 1ull);
          sv[k] = ok ? (own[k] + X[((1 - pair) * kHalf + k) * T + t]) * p.scale_log2 : -INFINITY;
        }
        if (j == 0) {
#pragma unroll
          for (int k = 0; k < kHalf; ++k) { m_ref[k] = sv[k]; l_part[k] = 0.f; }
          pair_reduce<kHalf, false>(m_ref, red, pair, wip, lane, rk);
          named_bar_sync(kBarVote, 128);   // keeps X reuse ordered like the vote below
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
              alpha[k] = (kMQ && mn == -INFINITY) ? 1.f : ex2_approx(m_ref[k] - mn);   // a row with no score yet
              m_ref[k] = mn;
              l_part[k] *= alpha[k];
            }
            if (wip == 0 && lane == 0) {
#pragma unroll
              for (int k = 0; k < kHalf; ++k) bc[pair * kHalf + k] = alpha[k];
            }
            named_bar_sync(kBarSm, 128);
            float alpha_all[NH];   // registers: the TMEM accesses below are compiler barriers
#pragma unroll
            for (int h = 0; h < NH; ++h) alpha_all[h] = bc[h];
            // rescale O^T (every head's column) after the previous tile's PV has landed
            wait(bar(C::bPDone + ((g - 1) & 1)), ((g - 1) >> 1) & 1);
            tc_fence_after();
            if (!aborted) {
#pragma unroll 1
              for (int mb = 0; mb < 4; ++mb) {
                uint32_t o[NH];
                const uint32_t ta = tmem + lane_off + C::kTmO + mb * NH;
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
        float pv[kHalf];
#pragma unroll
        for (int k = 0; k < kHalf; ++k) {
          // -inf scores give 0; so does a row with no score yet (m_ref -inf, multi-query)
          pv[k] = ex2_approx(sv[k] - ((kMQ && m_ref[k] == -INFINITY) ? 0.f : m_ref[k]));
          l_part[k] += pv[k];
        }
        if (g >= 2) wait(bar(C::bPDone + buf), ((g >> 1) - 1) & 1);
        if (!aborted) {
          // P^T[buf]: K-major, 128B swizzle; row = head, 64 tokens per 128-byte row
          uint8_t* pb = smem + C::kOffP + buf * C::kPBuf;
#pragma unroll
          for (int k = 0; k < kHalf; ++k) {
            const int h = pair * kHalf + k;
            const int off = (h >> 3) * 1024 + (h & 7) * 128 + ((((t >> 3) ^ (h & 7)) & 7) << 4) + (t & 7) * 2;
            *reinterpret_cast<__nv_bfloat16*>(pb + off) = __float2bfloat16_rn(pv[k]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(C::bPFull + buf));
        if (tid == 0) MLA_TRACE_EVENT(7, g);
      }
      // ------------------------------------------------------------ epilogue
      // The softmax sums and the LSE do not depend on O: they overlap the
      // item's last PV.  Then each 128-dim block of O^T is read from TMEM as
      // soon as its last MMA is done (PV order 0, 2, 1, 3), scaled by 1/l and
      // written through the warp's own staging rows (no CTA barrier).
      if (tid == 0 && nitem < 24) MLA_TRACE_RAW(15, 8 + 2 * nitem, clock64());
      const bool tid0 = tid == 0;
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
          if (kMQ)   // a row with nothing to attend: out 0
            *reinterpret_cast<float4*>(bc + pair * kHalf + k) = make_float4(
                l_tot[k] > 0.f ? __frcp_rn(l_tot[k]) : 0.f, l_tot[k + 1] > 0.f ? __frcp_rn(l_tot[k + 1]) : 0.f,
                l_tot[k + 2] > 0.f ? __frcp_rn(l_tot[k + 2]) : 0.f, l_tot[k + 3] > 0.f ? __frcp_rn(l_tot[k + 3]) : 0.f);
          else
            *reinterpret_cast<float4*>(bc + pair * kHalf + k) = make_float4(
                __frcp_rn(l_tot[k]), __frcp_rn(l_tot[k + 1]), __frcp_rn(l_tot[k + 2]), __frcp_rn(l_tot[k + 3]));
      }
      {
        // lane k of the pair's first warp writes head pair*kHalf + k
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
      float inv_l[NH];     // registers: the TMEM accesses below are compiler barriers
#pragma unroll
      for (int h = 0; h < NH; ++h) inv_l[h] = bc[h];
      if (tid == 0 && nitem < 8) MLA_TRACE_RAW(13, 8 * nitem, clock64());
      const bool st_bf16 = to_out && p.out_bf16;
      const int esz = st_bf16 ? 2 : 4;
      uint8_t* dst = to_out ? reinterpret_cast<uint8_t*>(p.out) + static_cast<size_t>(b) * p.heads * kLatent * esz
                            : reinterpret_cast<uint8_t*>(p.part_o + static_cast<size_t>(part) * p.heads * kLatent);
      uint8_t* wst = smem + C::kOffX + warp * NH * 32 * 4;   // this warp's [NH][32] staging rows
      const int lg = st_bf16 ? 2 : 3;                          // 16-byte chunks per head row: 4 or 8
#pragma unroll 1
      for (int r = 0; r < 2; ++r) {
        // blocks r and r+2 come from one latent unit; the commit after the
        // second also covers the first
        if (tid == 0 && nitem < 4) MLA_TRACE_RAW(14, 16 + 8 * nitem + r, clock64());
        wait(bar(C::bOBlk + r + 2), nitem & 1);
        if (tid == 0 && nitem < 4) MLA_TRACE_RAW(14, 48 + 4 * nitem + r, clock64());
        tc_fence_after();
        uint32_t o[2][NH];
        if (!aborted) {
          tmem_ld_cols<NH>(tmem + lane_off + C::kTmO + r * NH, o[0]);
          tmem_ld_cols<NH>(tmem + lane_off + C::kTmO + (r + 2) * NH, o[1]);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int h = 0; h < NH; ++h) o[0][h] = o[1][h] = 0;
        }
        if (r == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0 && !aborted) mbar_arrive(bar(C::bOEmpty));
        }
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int mb = r + 2 * hb;
          if (st_bf16) {
#pragma unroll
            for (int h = 0; h < NH; ++h)
              reinterpret_cast<__nv_bfloat16*>(wst)[h * 32 + lane] =
                  __float2bfloat16_rn(__uint_as_float(o[hb][h]) * inv_l[h]);
          } else {
#pragma unroll
            for (int h = 0; h < NH; ++h)
              reinterpret_cast<float*>(wst)[h * 32 + lane] = __uint_as_float(o[hb][h]) * inv_l[h];
          }
          __syncwarp();
          // the warp's block: NH heads x 32 dims as 16-byte chunks, head-major
#pragma unroll
          for (int k = 0; k < NH * 8 / 32; ++k) {
            const int c = lane + 32 * k;
            if (c < (NH << lg) && !aborted && part_ok) {
              const int h = c >> lg, cc = c & ((1 << lg) - 1);
              const uint4 v = *reinterpret_cast<const uint4*>(wst + (h * 32) * esz + 16 * cc);
              *reinterpret_cast<uint4*>(dst + (static_cast<size_t>(h) * kLatent + 128 * mb + 32 * warp) * esz + 16 * cc) =
                  v;
            }
          }
          __syncwarp();
        }
        if (tid == 0 && nitem < 8) MLA_TRACE_RAW(13, 8 * nitem + 1 + r, clock64());
      }
      named_bar_sync(kBarSm, 128);   // the staging rows double as the next tile's exchange buffer
      if (tid == 0 && nitem < 24) MLA_TRACE_RAW(15, 9 + 2 * nitem, clock64());
      ++nitem;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kPvWarp) tmem_dealloc(tmem, C::kTmemCols);
#ifdef MLA_TRACE
  if (threadIdx.x == 0) {
    MLA_TRACE_RAW(15, 1, static_cast<long long>(globaltimer()));
    MLA_TRACE_RAW(15, 4, clock64());
  }
#endif
}

template <int NH, bool kMQ>
int launch(const CUtensorMap& tm_kv, const CUtensorMap& tm_kr, const CUtensorMap& tm_qn, const CUtensorMap& tm_qr,
           const DecodeParams& p, int grid, cudaStream_t stream) {
  using C = Cfg<NH>;
  if (!set_smem_limit(reinterpret_cast<const void*>(&swab_kernel<NH, kMQ>), C::kSmemBytes)) return MLA_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // the prologue overlaps the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, swab_kernel<NH, kMQ>, tm_kv, tm_kr, tm_qn, tm_qr, p) != cudaSuccess)
    return MLA_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace swab

int launch_swab(int heads, const CUtensorMap& tm_kv, const CUtensorMap& tm_kr, const CUtensorMap& tm_qn,
                const CUtensorMap& tm_qr, const DecodeParams& p, int grid, cudaStream_t stream) {
  const bool mq = p.q_len > 1;
  if (heads == 16) return mq ? swab::launch<16, true>(tm_kv, tm_kr, tm_qn, tm_qr, p, grid, stream)
                             : swab::launch<16, false>(tm_kv, tm_kr, tm_qn, tm_qr, p, grid, stream);
  if (heads == 32) return mq ? swab::launch<32, true>(tm_kv, tm_kr, tm_qn, tm_qr, p, grid, stream)
                             : swab::launch<32, false>(tm_kv, tm_kr, tm_qn, tm_qr, p, grid, stream);
  return MLA_ERR_UNSUPPORTED;
}

}  // namespace mla
