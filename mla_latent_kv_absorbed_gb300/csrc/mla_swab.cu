// Absorbed MLA decode for few heads (H = 16 or 32) on sm_103a.
//
// With only 16 or 32 query heads the tensor core's M side cannot be the
// heads, so both products run "swapped": tokens (or latent dims) on M, heads
// on N.
//
//   QK:  S^T[64 tok x H]    = K_tile[64 tok x 576] . Q[H x 576]^T        (M = 64, K-major A and B)
//   PV:  O^T[128 dim x H]  += V^T[128 dim x 64 tok] . P^T[64 tok x H]    (M = 128, A read MN-major
//                                                                         from the same tile)
//
// The rows of a request are gathered from the page-size-1 cache with TMA
// gather4 (four slots per instruction) into 128-byte-swizzled "atoms" of 64
// tokens x 64 dims (8 KB): 8 latent atoms and 1 rope atom per 64-token tile.
// Latent atoms travel in pairs (16 KB ring units, the 128 latent dims one PV
// block consumes), one 32-lane gather4 instruction per unit.
// Each latent atom is read twice by the tensor core -- as part of the key
// (score over 576) and as the value (latent reused as V) -- and is released
// after its PV, so every cache byte crosses HBM once.
// ("实现差距：MLA 与 DeepSeek V3", section 2.4: dual-path score, FA2-style
// online softmax, kv_c reused as the value; "Attention backends", paragraph
// "MLA": 576 wide for k and 512 for v, one shared vector per token.)
//
// The shared-memory ring holds 2.75 (H=16) or 2.25 (H=32) tiles, so the gather of
// the next tile runs while the current one is scored.  A single warp issuing
// gather4 completes one op every ~70-110 cycles, so the tile's nine 16-op
// gather jobs are spread over several producer warps (nine with 16 heads,
// five with 32, whose softmax needs more registers per thread).
//
// Warp roles (one CTA per SM, persistent over the plan's work items):
//   warps 0-3   softmax / epilogue (TMEM lane quadrants 0-3)
//   warp 4      QK issuer and query loader (one thread, blocking waits)
//   warp 5      TMEM allocator and PV issuer (one thread, blocking waits)
//   warp 6      index stager: slot numbers to shared memory
//   warps 7..   gather producers
// With M = 64 the score tile S^T puts token rows 16q..16q+15 in TMEM lanes
// 32q..32q+15 (q = lane quadrant); O^T (M = 128) puts latent dim r in lane r.
//
// Softmax: scores are scaled into log2 units; each head keeps a reference
// maximum m_ref that only moves when a tile exceeds it by more than 8 (a
// group vote per tile); then O and the running sums are rescaled once.  So
// P = 2^(s - m_ref) <= 256 always fits bf16 and the fp32 sums.
#include "mla_device.cuh"
#include "mla_launch.h"

namespace mla {
namespace swab {

constexpr int kIdxSlots = 4;              // tiles of slot indices staged ahead
constexpr int kQkWarp = 4, kPvWarp = 5, kIdxWarp = 6, kProducerWarp0 = 7;

template <int NH>
struct Cfg {
  // Nine gather jobs per tile (latent atoms 0-7, the rope atom), 16 gather4
  // each; producer k takes jobs k, k + P, ...  With 16 heads every job has its
  // own warp; with 32 the softmax needs the registers of a smaller CTA.
  static constexpr int kProducers = (NH == 16) ? 9 : 5;
  static constexpr int kThreads = 32 * (kProducerWarp0 + kProducers);
  static constexpr int T = 64;                           // tokens per tile
  static constexpr int kPairSlots = (NH == 16) ? 11 : 9;  // ring of latent atom pairs (16 KB each)
  static constexpr int kRopeSlots = 3;
  static constexpr int kAtom = T * 128;                  // 8 KB: 64 tokens x 64 dims
  static constexpr int kPair = 2 * kAtom;                // dims 128u .. 128u+127
  static constexpr int kQAtom = NH * 128;
  static constexpr int kQBytes = 9 * kQAtom;
  static constexpr int kPBytes = NH * 128;               // P^T: NH heads x 64 tokens
  static constexpr int kOffLat = 0;
  static constexpr int kOffRope = kOffLat + kPairSlots * kPair;
  static constexpr int kOffQ = kOffRope + kRopeSlots * kAtom;
  static constexpr int kOffP = kOffQ + kQBytes;
  static constexpr int kOffRed = kOffP + 2 * kPBytes;    // [2][4][NH] floats
  static constexpr int kOffBar = kOffRed + 2 * 4 * NH * 4;
  // barrier indices
  static constexpr int bLatFull = 0;
  static constexpr int bLatEmpty = kPairSlots;
  static constexpr int bRopeFull = 2 * kPairSlots;
  static constexpr int bRopeEmpty = bRopeFull + kRopeSlots;
  static constexpr int bQFull = bRopeEmpty + kRopeSlots;
  static constexpr int bQEmpty = bQFull + 1;
  static constexpr int bSFull = bQEmpty + 1;
  static constexpr int bSEmpty = bSFull + 2;
  static constexpr int bPFull = bSEmpty + 2;
  static constexpr int bPEmpty = bPFull + 2;
  static constexpr int bPvDone = bPEmpty + 2;
  static constexpr int bOFull = bPvDone + 1;
  static constexpr int bOEmpty = bOFull + 1;
  static constexpr int bDrain = bOEmpty + 1;             // both issuers' final commits
  static constexpr int bIdxFull = bDrain + 1;
  static constexpr int bIdxEmpty = bIdxFull + kIdxSlots;
  static constexpr int kNumBars = bIdxEmpty + kIdxSlots;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffLast = kOffMisc + 16;           // [kPairSlots + kRopeSlots] ints
  static constexpr int kOffIdx = (kOffLast + 4 * (kPairSlots + kRopeSlots) + 15) / 16 * 16;   // [kIdxSlots][T] ints
  static constexpr int kSmemBytes = kOffIdx + 4 * kIdxSlots * T + 1024;   // + alignment slack
  static constexpr int kTmemCols = (6 * NH <= 128) ? 128 : 256;
  static constexpr int kTmS = 0;       // S^T buffers: columns [0,NH) and [NH,2NH)
  static constexpr int kTmO = 2 * NH;  // O^T blocks: columns 2NH + mb*NH
  static constexpr uint32_t kIdescQK = idesc_bf16(64, NH, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16(128, NH, true, false);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "atoms must be 1024-byte aligned");
  static_assert(kOffIdx % 16 == 0, "index ring alignment");
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

// A tile is five ring units: latent atom pairs u = 0..3 (dims 128u..128u+127,
// 16 KB) and the rope atom u = 4 (8 KB).  Returns the unit's ring position.
struct UnitRef {
  uint32_t addr, full, empty, use, slot;
  bool rope;
};

template <int NH>
__device__ __forceinline__ UnitRef unit_ref(uint32_t base, uint32_t g, int u) {
  using C = Cfg<NH>;
  UnitRef r;
  if (u < 4) {
    const uint32_t seq = g * 4 + u;
    r.slot = seq % C::kPairSlots;
    r.use = seq / C::kPairSlots;
    r.addr = base + C::kOffLat + r.slot * C::kPair;
    r.full = base + C::kOffBar + 8u * (C::bLatFull + r.slot);
    r.empty = base + C::kOffBar + 8u * (C::bLatEmpty + r.slot);
    r.rope = false;
  } else {
    r.slot = g % C::kRopeSlots;
    r.use = g / C::kRopeSlots;
    r.addr = base + C::kOffRope + r.slot * C::kAtom;
    r.full = base + C::kOffBar + 8u * (C::bRopeFull + r.slot);
    r.empty = base + C::kOffBar + 8u * (C::bRopeEmpty + r.slot);
    r.rope = true;
  }
  return r;
}

template <int NH>
__global__ void __launch_bounds__(Cfg<NH>::kThreads, 1)
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
  int* last_armed = reinterpret_cast<int*>(smem + C::kOffLast);   // per ring slot: last armed use
  const WaitCtx wc{abort_flag, p.status};

  const int w = blockIdx.x;
  const int32_t* wptr = p.plan + kHeaderWords;
  const int it0 = wptr[w], it1 = wptr[w + 1];
  const int32_t* items = p.plan + p.items_off;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kPairSlots; ++i) { mbar_init(bar(C::bLatFull + i), 1); mbar_init(bar(C::bLatEmpty + i), 1); }
    for (int i = 0; i < C::kRopeSlots; ++i) { mbar_init(bar(C::bRopeFull + i), 1); mbar_init(bar(C::bRopeEmpty + i), 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::bSFull + i), 1); mbar_init(bar(C::bSEmpty + i), 4);
      mbar_init(bar(C::bPFull + i), 4); mbar_init(bar(C::bPEmpty + i), 1);
    }
    mbar_init(bar(C::bQFull), 1); mbar_init(bar(C::bQEmpty), 1);
    mbar_init(bar(C::bPvDone), 1); mbar_init(bar(C::bOFull), 1); mbar_init(bar(C::bOEmpty), 4);
    mbar_init(bar(C::bDrain), 2);
    for (int i = 0; i < kIdxSlots; ++i) { mbar_init(bar(C::bIdxFull + i), 1); mbar_init(bar(C::bIdxEmpty + i), C::kProducers); }
    for (int i = 0; i < C::kPairSlots + C::kRopeSlots; ++i) last_armed[i] = -1;
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

  if (warp == kIdxWarp) {
    // ---------------------------------------------------------- index stager
    // Walks the tiles in plan order, loads each tile's 64 slot numbers
    // (coalesced), replaces out-of-range ones by slot 0 (flagged) and the
    // ragged tail by the last valid slot, and publishes them in a small ring.
    int* idx_ring = reinterpret_cast<int*>(smem + C::kOffIdx);
    uint32_t g = 0;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
      if (!item_ok(p, b, s, e)) {
        if (lane == 0) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
        continue;
      }
      const int n = e - s;
      for (int t0 = 0; t0 < n; t0 += C::T, ++g) {
        const uint32_t slot = g % kIdxSlots, use = g / kIdxSlots;
        int v[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) v[k] = __ldg(p.kv_indices + s + min(t0 + lane + 32 * k, n - 1));
        bool w_ok = true;
        if (lane == 0 && use > 0) w_ok = mbar_wait(bar(C::bIdxEmpty + slot), (use - 1) & 1, wc);
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) { ok = false; break; }
        bool oob = false;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          if (v[k] < 0 || static_cast<long long>(v[k]) >= p.num_slots) { oob = true; v[k] = 0; }
          idx_ring[slot * C::T + lane + 32 * k] = v[k];
        }
        if (__any_sync(0xffffffffu, oob) && lane == 0) record_status(p.status, MLA_ERR_INDEX_OOB);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::bIdxFull + slot));
      }
    }
  } else if (warp >= kProducerWarp0) {
    // ------------------------------------------------------ gather producers
    // A warp completes one gather4 only every ~70-110 cycles, so a tile's
    // landing time is set by how many gathers one warp issues for it.  The
    // tile's nine jobs (latent atoms 0-7, the rope atom; 16 gather4 each) are
    // dealt round-robin over the producers.  A pair unit is armed by the
    // producer of its even atom.
    const int pw = warp - kProducerWarp0;
    if (lane == 0 && pw == 0) tma_prefetch_desc(&tm_kv);
    const uint64_t pol = l2_policy_evict_first();
    const int* idx_ring = reinterpret_cast<const int*>(smem + C::kOffIdx);
    uint32_t g = 0;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
      if (!item_ok(p, b, s, e)) continue;
      const int n = e - s;
      for (int t0 = 0; t0 < n && ok; t0 += C::T, ++g) {
        const uint32_t islot = g % kIdxSlots;
        bool w_ok = true;
        if (lane == 0) w_ok = mbar_wait(bar(C::bIdxFull + islot), (g / kIdxSlots) & 1, wc);
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) { ok = false; break; }
        // lane l < 16 holds tokens 4l..4l+3 (gather op l of an atom)
        const int4 v = *reinterpret_cast<const int4*>(idx_ring + islot * C::T + 4 * (lane & 15));
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::bIdxEmpty + islot));
        if (lane == 0) MLA_TRACE_EVENT(pw == 0 ? 0 : (pw < 4 ? 8 + pw : 15), g);
#pragma unroll 1
        for (int a = pw; a < 9 && ok; a += C::kProducers) {
          const UnitRef r = unit_ref<NH>(base, g, a < 8 ? a >> 1 : 4);
          bool e_ok = true;
          if (lane == 0 && r.use > 0) e_ok = mbar_wait(r.empty, (r.use - 1) & 1, wc);
          e_ok = __shfl_sync(0xffffffffu, e_ok, 0);
          if (!e_ok) { ok = false; break; }
          const bool arms = r.rope || (a & 1) == 0;
          if (lane == 0 && arms) mbar_arrive_expect_tx(r.full, r.rope ? C::kAtom : C::kPair);
          __syncwarp();
          if (lane < 16)
            tma_gather4(r.addr + (r.rope ? 0 : (a & 1) * C::kAtom) + lane * 512, &tm_kv, 64 * a, v.x, v.y, v.z,
                        v.w, r.full, pol);
          if (lane == 0) atomicMax(last_armed + (r.rope ? C::kPairSlots : 0) + r.slot, static_cast<int>(r.use));
        }
        if (lane == 0 && pw == 0) MLA_TRACE_EVENT(1, g);
      }
    }
    // drain: every copy armed by any producer has landed before the CTA can
    // exit (slots are shared between producer warps, so use the latest use)
    named_bar_sync(3, 32 * C::kProducers);
    if (pw == 0) {
      for (int i = lane; i < C::kPairSlots + C::kRopeSlots; i += 32) {
        const int u = last_armed[i];
        const int bfull = i < C::kPairSlots ? C::bLatFull + i : C::bRopeFull + (i - C::kPairSlots);
        if (u >= 0) drain_wait(bar(bfull), u & 1);
      }
    }
    __syncwarp();
  } else if (warp == kQkWarp) {
    // ----------------------------------------------- QK issuer + query loader
    // One thread that blocks on its barriers (no polling).  Per item it loads
    // the query (latent atoms and rope) once the previous item's last QK has
    // read the old one; per tile it scores each ring unit as it lands.
    if (lane == 0) {
      tma_prefetch_desc(&tm_qn);
      tma_prefetch_desc(&tm_qr);
      const uint64_t dq = sdesc(base + C::kOffQ, 16, 1024);        // Q atom 0 (B of QK)
      const uint64_t dk = sdesc(base + C::kOffLat, 16, 1024);      // pair slot 0 (A of QK)
      const uint64_t dr = sdesc(base + C::kOffRope, 16, 1024);     // rope slot 0 (A of QK)
      auto D = [](uint64_t d, uint32_t byte_off) -> uint64_t { return d + (byte_off >> 4); };
      const uint32_t qbase = base + C::kOffQ;
      uint32_t g = 0, nitem = 0, qs = 0, qph = 0, qr = 0, qrph = 0;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
        if (!item_ok(p, b, s, e)) continue;
        const int nt = (e - s + C::T - 1) / C::T;
        if (nitem > 0 && !mbar_wait(bar(C::bQEmpty), (nitem - 1) & 1, wc)) break;
        mbar_arrive_expect_tx(bar(C::bQFull), C::kQBytes);
        for (int a = 0; a < 8; ++a) tma_load_2d(qbase + a * C::kQAtom, &tm_qn, 64 * a, b * p.heads, bar(C::bQFull));
        tma_load_2d(qbase + 8 * C::kQAtom, &tm_qr, 0, b * p.heads, bar(C::bQFull));
        if (!mbar_wait(bar(C::bQFull), nitem & 1, wc)) break;
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t d_s = tmem + C::kTmS + (g & 1) * NH;
          if (g >= 2 && !mbar_wait(bar(C::bSEmpty + (g & 1)), ((g >> 1) - 1) & 1, wc)) { ok = false; break; }
          MLA_TRACE_EVENT(2, g);
#pragma unroll 1
          for (int u = 0; u < 4 && ok; ++u) {
            if (!mbar_wait(bar(C::bLatFull + qs), qph, wc)) { ok = false; break; }
            tc_fence_after();
            const uint64_t ak = D(dk, qs * C::kPair);
            const uint64_t bq = D(dq, 2 * u * C::kQAtom);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_ss(d_s, D(ak, h * C::kAtom + 32 * kk), D(bq, h * C::kQAtom + 32 * kk), C::kIdescQK,
                        (u | h | kk) != 0 ? 1u : 0u);
            if (++qs == static_cast<uint32_t>(C::kPairSlots)) { qs = 0; qph ^= 1; }
          }
          if (!ok || !mbar_wait(bar(C::bRopeFull + qr), qrph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ar = D(dr, qr * C::kAtom);
          const uint64_t bq = D(dq, 8 * C::kQAtom);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) umma_ss(d_s, D(ar, 32 * kk), D(bq, 32 * kk), C::kIdescQK, 1u);
          umma_commit(bar(C::bRopeEmpty + qr));
          if (++qr == static_cast<uint32_t>(C::kRopeSlots)) { qr = 0; qrph ^= 1; }
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
    // Issues a tile's PV once its P^T is written and releases each pair unit
    // as soon as its 128-dim block is done.
    if (lane == 0) {
      const uint64_t dv = sdesc(base + C::kOffLat, C::kAtom, 1024);  // pair slot 0 (A of PV, MN-major)
      const uint64_t dp = sdesc(base + C::kOffP, 16, 1024);        // P^T buffer 0 (B of PV)
      auto D = [](uint64_t d, uint32_t byte_off) -> uint64_t { return d + (byte_off >> 4); };
      uint32_t g = 0, nitem = 0, ps = 0;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
        if (!item_ok(p, b, s, e)) continue;
        const int nt = (e - s + C::T - 1) / C::T;
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t buf = g & 1;
          if (!mbar_wait(bar(C::bPFull + buf), (g >> 1) & 1, wc)) { ok = false; break; }
          if (j == 0 && nitem > 0 && !mbar_wait(bar(C::bOEmpty), (nitem - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          MLA_TRACE_EVENT(4, g);
          const uint64_t bp = D(dp, buf * C::kPBytes);
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
            const uint64_t av = D(dv, ps * C::kPair);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_ss(tmem + C::kTmO + mb * NH, D(av, ks * 2048), D(bp, ks * 32), C::kIdescPV,
                      (j == 0 && ks == 0) ? 0u : 1u);
            umma_commit(bar(C::bLatEmpty + ps));
            ps = (ps + 1 == static_cast<uint32_t>(C::kPairSlots)) ? 0 : ps + 1;
          }
          umma_commit(bar(C::bPEmpty + buf));
          umma_commit(bar(C::bPvDone));
          if (j == nt - 1) umma_commit(bar(C::bOFull));
          MLA_TRACE_EVENT(5, g);
        }
        ++nitem;
      }
      umma_commit(bar(C::bDrain));
      drain_wait(bar(C::bDrain), 0);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------- softmax + epilogue
    const int wq = warp;                          // lane quadrant
    const int t = 16 * wq + lane;                 // token row of S^T (lanes 0-15 only)
    const bool row_lane = lane < 16;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int dim_row = 32 * wq + lane;           // latent row of O^T (within a 128-dim block)
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
        if (threadIdx.x == 0) MLA_TRACE_EVENT(6, g);
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
        const bool valid = row_lane && t < n - j * C::T;
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
        if (!aborted && row_lane) {
          // P^T[buf]: K-major, 128B swizzle; row = head, 64 tokens per 128-byte row
          uint8_t* pb = smem + C::kOffP + buf * C::kPBytes;
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const int off = (h >> 3) * 1024 + (h & 7) * 128 + ((((t >> 3) ^ (h & 7)) & 7) << 4) + (t & 7) * 2;
            *reinterpret_cast<__nv_bfloat16*>(pb + off) = __float2bfloat16_rn(pv[h]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(C::bPFull + buf));
        if (threadIdx.x == 0) MLA_TRACE_EVENT(7, g);
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
          const int dim = 128 * mb + dim_row;
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
        const int tid = threadIdx.x;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          if (tid == h) {
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
  if (warp == kPvWarp) tmem_dealloc(tmem, C::kTmemCols);
}

template <int NH>
int launch(const CUtensorMap& tm_kv, const CUtensorMap& tm_qn, const CUtensorMap& tm_qr,
           const DecodeParams& p, int grid, cudaStream_t stream) {
  using C = Cfg<NH>;
  static bool attr_done = false;   // the attribute is per function, set once per process
  if (!attr_done) {
    if (cudaFuncSetAttribute(swab_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return MLA_ERR_CUDA;
    attr_done = true;
  }
  swab_kernel<NH><<<grid, C::kThreads, C::kSmemBytes, stream>>>(tm_kv, tm_qn, tm_qr, p);
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace swab

int launch_swab(int heads, const CUtensorMap& tm_kv, const CUtensorMap& tm_qn,
                const CUtensorMap& tm_qr, const DecodeParams& p, int grid, cudaStream_t stream) {
  if (heads == 16) return swab::launch<16>(tm_kv, tm_qn, tm_qr, p, grid, stream);
  if (heads == 32) return swab::launch<32>(tm_kv, tm_qn, tm_qr, p, grid, stream);
  return MLA_ERR_UNSUPPORTED;
}

}  // namespace mla
