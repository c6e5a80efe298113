// Absorbed MLA decode over an FP8 (E4M3) latent cache for many heads
// (H = 48..128, step 16) on sm_103a: the two-CTA design of the bf16 kernel
// (mla_pair.cu) with 8-bit operands on the tensor core (tcgen05.mma
// kind::f8f6f4, K = 32 per instruction) and no dequantisation pass.
// ("MLA and torch.compile: v0.3's two sources", section "MLA: starting from a
// 439-line commit": the FP8 KV cache; "实现差距：MLA 与 DeepSeek V3", section
// 2.4: the latent and rope dot products summed and scaled, FA2-style online
// softmax, the latent rows reused as the values.)
//
// As in the bf16 kernel a worker is a cluster of two CTAs, CTA c owning latent
// dims [256c, 256c+256) and rope dims [32c, 32c+32); partial scores are
// exchanged as 23-bit fixed point (error at most 2^-22 of the half row's
// largest partial, at any query magnitude), and each CTA adds its own exact
// partial to the peer's decoded one and normalises its half of O with its own
// row sum.  What changes is the arithmetic of the two products:
//   - the cache rows stay E4M3 (value = code x kv_scale);
//   - the query is carried as two 8-bit parts: per head, q' = q * 2^a with the
//     power of two a that puts max |q'| over this CTA's 288 dims in [128, 256),
//     hi = e4m3(q'), lo = e5m2(q' - hi).  The residual of a bf16 value after
//     its 4 leading bits has at most 3 significant bits, which E5M2 holds, and
//     its range reaches 2^-16, so hi + lo is q' exactly for |q'| >= 2^-6 (an
//     E4M3 lo, unscaled in the shared accumulator, would lose the bits of
//     every element below 2^-2: about 2e-6 of the row's largest partial).
//     Both parts are A operands from TMEM (4 codes per column; the lo MMAs
//     take A as E5M2, B as E4M3) and accumulate into the same scores, so each
//     latent K-step of 32 dims takes 2 MMAs (the bf16 kernel takes 2 of 16);
//     partials are multiplied by 2^-a (the senders' before quantising, the
//     softmax warps' own before adding the peer's), so the two CTAs' partials
//     are in the same units;
//   - P' = 2^(s - m_ref + 5) likewise (a reference that lags the maximum by at
//     most 3, so P' <= 256 and the maximum's weight is >= 32): hi = e4m3(P'), lo = e4m3(P' - hi),
//     written side by side in the exchange slot's 128-byte rows (bytes 0-63
//     hi, 64-127 lo, one byte per token): 2 MMAs per 32-token K-step (the
//     split takes the difference in f16: five instructions per pair).
// hi + lo holds P to about 8 significant bits (bf16 has 8), within 2^-10
// absolute for the small weights.  The epilogue multiplies O by
// kv_scale / l; the score decode multiplies by sm_scale * log2(e) * kv_scale.
//
// TMEM (512 columns per CTA): O_c [0,256) fp32; the query's hi part [256,320)
// and lo part [320,384) (4 codes per column); two score buffers [384,512).
//
// Shared memory per CTA: a ring of 8 latent blocks (64 tokens x 256 dims,
// 16 KB: two 128-dim atoms, 128-byte swizzle), 4 rope atoms (64 tokens x 32
// dims, 2 KB, 32-byte swizzle), the rope query's hi and lo parts (128 rows x
// 32 bytes each, 32-byte swizzle), 3 exchange slots (the high parts of the
// peer's codes, then P), their low-byte blocks, the peer's exponents, the
// softmax warps' reduction buffers and the CTA's first work items.
//
// Warp roles per CTA (736 threads), as in the bf16 kernel:
//   warps 8-15  senders: at an item's start, load the head's query dims of
//               this CTA, scale and split them into TMEM (latent) and shared
//               memory (rope); per tile, quantise their part of the partial
//               and push the codes
//   warps 0-7   softmax: add the peer's decoded partial to this CTA's, softmax, P (hi and lo) over the
//               peer's rows; the epilogue
//   warp 16     QK issuer (one thread)
//   warp 17     TMEM allocator and PV issuer (one thread)
//   warps 18-22 gather producers: latent atom (pw >> 1) x token half (pw & 1)
//               for pw < 4 (8 gather4 of 128-byte rows each), the rope (16
//               gather4 of 32-byte rows)
#include "mla_device.cuh"
#include "mla_launch.h"

namespace mla {
namespace pair8 {

constexpr int T = 64;                        // tokens per tile
constexpr int TH = 32;                       // tokens of a tile per row warp
constexpr int kRowWarps = 8;                 // softmax warps 0-7 and sender warps 8-15 alike
constexpr int kProducers = 5;                // latent atoms 0-3 and the rope
constexpr int kSendWarp0 = 8, kMmaWarp = 16, kLoaderWarp = 17, kProducerWarp0 = 18;
constexpr int kThreads = 32 * (kProducerWarp0 + kProducers);
// A latent block is held from its gathers until its PV, the whole life of a
// tile in the pipeline, so the ring is as deep as shared memory allows.
constexpr int kLatBlocks = 8;                // ring of latent blocks (every latent producer fills every block)
constexpr int kRopeSlots = 4;               // a rope slot is free again once QK has read it
constexpr int kXSlots = 3;                   // exchange slots
constexpr int kLead = 6;                     // a producer issues tile g once tile g - kLead has landed
constexpr int kRopeLead = kLead < kRopeSlots ? kLead : kRopeSlots;   // the same for the rope
constexpr int kAtom = T * 128;               // 8 KB: 64 tokens x 128 E4M3 dims
constexpr int kLatBlock = 2 * kAtom;         // 16 KB: 64 tokens x 256 dims
constexpr int kRopeAtom = T * 32;            // 2 KB: 64 tokens x this CTA's 32 rope dims (32-byte swizzle)
constexpr int kQRPlane = 128 * 32;           // rope query part: 128 rows x 32 E4M3 (32-byte swizzle)
constexpr int kQRBytes = 2 * kQRPlane;       // hi, then lo
constexpr int kXSlot = 128 * 128;            // 128 rows x 128 B (64 int16 scores, then P: 64 hi and 64 lo E4M3)
constexpr int kXLoSlot = 128 * 64;           // the codes' low bytes: [4 chunks (half, part)][128 rows] x 16 B
constexpr int kXeSlot = 2 * 128 * 4;         // [2 token halves][128 rows] int32 exponents
constexpr int kXBytes = kXSlot + kXLoSlot + kXeSlot;   // bytes the peer sends per tile
constexpr int kOffLat = 0;
constexpr int kOffRope = kOffLat + kLatBlocks * kLatBlock;
constexpr int kOffQR = kOffRope + kRopeSlots * kRopeAtom;   // rope query hi | lo (K-major SW32)
constexpr int kOffX = kOffQR + kQRBytes;
constexpr int kOffXLo = kOffX + kXSlots * kXSlot;       // [kXSlots] low-byte blocks from the peer
constexpr int kOffXE = kOffXLo + kXSlots * kXLoSlot;    // [kXSlots] exponent blocks from the peer
constexpr int kOffRed = kOffXE + kXSlots * kXeSlot;     // [2 bufs][2 halves][128] row maxima, [2][128] row sums
constexpr int kOffBar = kOffRed + (2 * 2 * 128 + 2 * 128) * 4;
// barriers
constexpr int bLatFull = 0;
constexpr int bLatEmpty = bLatFull + kLatBlocks;
constexpr int bRopeFull = bLatEmpty + kLatBlocks;
constexpr int bRopeEmpty = bRopeFull + kRopeSlots;
constexpr int bQFull = bRopeEmpty + kRopeSlots;
constexpr int bQEmpty = bQFull + 1;
constexpr int bSFull = bQEmpty + 1;          // [2] this CTA's partial is in the S buffer
constexpr int bSFree = bSFull + 2;           // [2] the senders and the softmax warps have read the S buffer
constexpr int bPFull = bSFree + 2;           // [kXSlots] P is in the exchange slot
constexpr int bPvDone = bPFull + kXSlots;    // [2] PV(g) has completed (buffer g mod 2)
constexpr int bOFull = bPvDone + 2;
constexpr int bOEmpty = bOFull + 1;
constexpr int bXFull = bOEmpty + 1;          // [kXSlots] the peer's rows have landed in this CTA's slot
constexpr int bXFree = bXFull + kXSlots;     // [kXSlots] the PEER's slot may take this CTA's next rows
constexpr int bDrain = bXFree + kXSlots;
constexpr int kNumBars = bDrain + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffLast = kOffMisc + 16;      // [kLatBlocks + kRopeSlots] last armed use
constexpr int kItemCache = 64;              // this CTA's first work items, copied to shared memory
constexpr int kOffItems = (kOffLast + 4 * (kLatBlocks + kRopeSlots) + 15) / 16 * 16;
constexpr int kSmemBytes = kOffItems + 16 * kItemCache + 1024;
constexpr int kTmO = 0, kTmQHi = 256, kTmQLo = 320, kTmS = 384;
constexpr uint32_t kIdescQK = idesc_e4m3(128, T, false, false);     // M=128 heads, N=64 tokens
constexpr uint32_t kIdescQKLo = idesc_f8(kFmtE5M2, kFmtE4M3, 128, T, false, false);   // the query's E5M2 low part
constexpr uint32_t kIdescPV = idesc_e4m3(128, 256, false, true);    // N=256 dims, B (V) MN-major
static_assert(kProducers == 5, "producers 0-3 gather the latent atoms, producer 4 the rope");
static_assert(kThreads == 736, "23 warps");
static_assert(kLead < kLatBlocks && kRopeLead <= kRopeSlots, "a ring slot's phase must not be lapped while waited on");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kXSlots <= 3, "the rescale's wait on PV(g-1) relies on PV(g-3) being complete");
static_assert(kOffRope % 1024 == 0 && kOffQR % 1024 == 0 && kOffX % 1024 == 0 && kXSlot % 1024 == 0 &&
                  kOffXE % 16 == 0 && kOffBar % 8 == 0,
              "alignment");

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

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > MLA_WAIT_LIMIT_NS) return;
  }
}

// 2^k as a float, for -126 <= k <= 127.
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float(static_cast<uint32_t>(k + 127) << 23); }

// Partial scores travel as 23-bit fixed point with a power-of-two step per
// row and 32-token half: with e the exponent of the half row's largest
// |partial| (nudged up by 2^-21 so that no code reaches 2^22), the step is
// 2^(e-21), so a code q = rint(partial / step) has |q| < 2^22 and the
// rounding error is at most 2^-22 of the largest |partial|, about fp32's own
// rounding of a sum of 288 products.  The code goes as offset binary
// u = q + 2^22 in 23 bits: its high 16 bits (u >> 8) in the slot's 128-byte
// rows (the bytes P later overwrites in place), its low 8 bits in a side
// block.  Rounding and decoding use full-rate float arithmetic:
//   encode: partial / step + 1.5 * 2^23 rounds to the nearest integer (ties to
//           even) and leaves u in the low 23 bits of the float;
//   decode: the bits 0x4B000000 | x are the float 2^23 + x, so with
//           fh = 2^23 + (u >> 8) and fl = 2^23 + (u & 255),
//           fh * 256 step + fl * step - (2^31 + 2^23 + 2^22) step = q * step,
//           exactly, as two FMAs whose results are representable.
// The receiver forms q * step exactly from the peer's codes, adds it to its
// own exact partial and multiplies the sum by the score scale once.  The two
// CTAs' scores may then differ in their last bits (each rounds only the
// other's partial); that is harmless, as each CTA normalises its own half of
// O with row sums of its own scores.
constexpr float kEncBias = 12582912.0f;      // 1.5 * 2^23
constexpr float kDecHi = 2160066560.0f;      // 2^31 + 2^23 + 2^22 = 515 * 2^22 (exact in fp32)

__global__ void __launch_bounds__(kThreads, 1)
    pair8_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_kr,
                 const DecodeParams p, const float kv_scale) {
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
#ifdef MLA_TRACE
  if (threadIdx.x == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    MLA_TRACE_RAW(15, 0, static_cast<long long>(globaltimer()));
    MLA_TRACE_RAW(15, 2, static_cast<long long>(smid));
    MLA_TRACE_RAW(15, 3, clock64());
  }
#endif

  const int w = blockIdx.x >> 1;
  const int H = p.heads;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kLatBlocks; ++i) { mbar_init(bar(bLatFull + i), 1); mbar_init(bar(bLatEmpty + i), 1); }
    for (int i = 0; i < kRopeSlots; ++i) { mbar_init(bar(bRopeFull + i), 1); mbar_init(bar(bRopeEmpty + i), 1); }
    mbar_init(bar(bQFull), kRowWarps);           // the sender warps (latent parts in TMEM, rope parts in smem)
    mbar_init(bar(bQEmpty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bSFull + i), 1); mbar_init(bar(bSFree + i), 2 * kRowWarps);
    }
    for (int i = 0; i < kXSlots; ++i) {
      mbar_init(bar(bPFull + i), kRowWarps);
      mbar_init(bar(bXFull + i), 1);             // own expect_tx; the bytes come from the peer
      mbar_init(bar(bXFree + i), 1);             // the peer's PV commit
    }
    mbar_init(bar(bPvDone), 1);
    mbar_init(bar(bPvDone + 1), 1);
    mbar_init(bar(bOFull), 1);
    mbar_init(bar(bOEmpty), kRowWarps);
    mbar_init(bar(bDrain), 2);                   // both issuers' final commits
    for (int i = 0; i < kLatBlocks + kRopeSlots; ++i) last_armed[i] = -1;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kLoaderWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  cluster_sync_all();                            // both CTAs' barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // launched as a programmatic dependent of the previous kernel in the
  // stream: everything above overlapped its tail; its results (the plan,
  // indices, query, cache rows) are read only after it has finished
  griddep_wait();
  int it0, it1;
  plan_items(p, w, it0, it1);
  const int32_t* items = p.plan + p.items_off;
  // this CTA's first kItemCache items, read once: no warp waits on the plan
  // in global memory at an item start
  int32_t* s_items = reinterpret_cast<int32_t*>(smem + kOffItems);
  const int n_cached = min(max(it1 - it0, 0), kItemCache);
  for (int i = threadIdx.x; i < 4 * n_cached; i += blockDim.x) s_items[i] = items[4 * it0 + i];
  __syncthreads();
  auto item_w = [&](int it, int k) -> int {
    return it - it0 < kItemCache ? s_items[4 * (it - it0) + k] : items[4 * it + k];
  };
  const int nnz = __ldg(p.kv_indptr + p.batch);
  // the merge kernel may be launched now: it waits for this grid to finish
  griddep_launch_dependents();
  bool aborted = false;                          // set by the softmax / sender warps only

  if (warp >= kProducerWarp0) {
    // ------------------------------------------------------ gather producers
    // Producer pw < 4 gathers latent atom pw >> 1 (128 dims of the CTA's
    // half) for token half pw & 1 (lanes 0-7: 8 gather4 of 128-byte rows);
    // producer 4 gathers the CTA's 32 rope dims of every token (lanes 0-15:
    // 16 gather4 of 32-byte rows).  Each loads its tile's slot numbers before
    // it waits for ring space; an out-of-range slot reads row 0 and sets
    // MLA_ERR_INDEX_OOB, the ragged tail repeats the last valid slot.
    const int pw = warp - kProducerWarp0;
    if (lane == 0 && pw == 0) tma_prefetch_desc(&tm_kv);
    if (lane == 0 && pw == 4) tma_prefetch_desc(&tm_kr);
    const uint64_t pol = l2_policy_evict_first();
    // The slot numbers of the next tile are loaded while this tile waits for
    // ring space and issues its gathers, so their latency is hidden.
    int it = it0, s = 0, n = 0;
    auto next_item = [&]() {                     // first usable item from `it` on
      for (; it < it1; ++it) {
        const int b = item_w(it, 0), s0 = item_w(it, 1), e = item_w(it, 2);
        if (item_ok(p, nnz, b, s0, e)) {
          if (pw == 0 && lane == 0 && !item_in_request(p, b, s0, e)) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
          s = s0;
          n = e - s0;
          return;
        }
        if (lane == 0 && pw == 0) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
      }
    };
    const int grp = pw < 4 ? 8 * (pw & 1) + (lane & 7) : (lane & 15);   // group of 4 tokens in the tile
    const bool active = pw < 4 ? lane < 8 : lane < 16;
    auto load_slots = [&](int t0, int (&v)[4]) {
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = __ldg(p.kv_indices + s + min(t0 + 4 * grp + k, n - 1));
    };
    next_item();
    int t0 = 0;
    int vn[4] = {0, 0, 0, 0};
    if (it < it1) load_slots(0, vn);
    uint32_t g = 0;
    bool ok = true;
    while (it < it1 && ok) {
      int v[4];
      bool oob = false;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[k] = vn[k];
        if (v[k] < 0 || static_cast<long long>(v[k]) >= p.num_slots) { oob = true; v[k] = 0; }
      }
      if (oob && pw == 4) record_status(p.status, MLA_ERR_INDEX_OOB);   // the rope producer sees every token
      // advance the cursor and prefetch the next tile's slot numbers
      t0 += T;
      if (t0 >= n) {
        ++it;
        next_item();
        t0 = 0;
      }
      if (it < it1) load_slots(t0, vn);
      if (lane == 0 && pw == 0) MLA_TRACE_EVENT(0, g);
      {
        const bool rope = pw == 4;
        const uint32_t nslots = rope ? kRopeSlots : kLatBlocks;
        const uint32_t slot = g % nslots, use = g / nslots;
        const uint32_t full = bar((rope ? bRopeFull : bLatFull) + slot);
        bool e_ok = true;
        if (lane == 0 && use > 0) e_ok = mbar_wait(bar((rope ? bRopeEmpty : bLatEmpty) + slot), (use - 1) & 1, wc);
        const uint32_t lead = rope ? kRopeLead : kLead;
        if (lane == 0 && e_ok && g >= lead) {   // pace: tile g - lead has landed
          const uint32_t gp = g - lead;
          e_ok = mbar_wait(bar((rope ? bRopeFull : bLatFull) + gp % nslots), (gp / nslots) & 1, wc);
        }
        e_ok = __shfl_sync(0xffffffffu, e_ok, 0);
        if (!e_ok) { ok = false; break; }
        if (rope) {
          if (lane == 0) mbar_arrive_expect_tx(full, kRopeAtom);
          if (lane == 0) MLA_TRACE_EVENT(11, g);
          __syncwarp();
          if (active)
            tma_gather4(base + kOffRope + slot * kRopeAtom + grp * 128, &tm_kr, 512 + 32 * static_cast<int>(cta),
                        v[0], v[1], v[2], v[3], full, pol);
          if (lane == 0) atomicMax(last_armed + kLatBlocks + slot, static_cast<int>(use));
        } else {
          if (lane == 0 && pw == 0) mbar_arrive_expect_tx(full, kLatBlock);
          __syncwarp();
          if (active)
            tma_gather4(base + kOffLat + slot * kLatBlock + (pw >> 1) * kAtom + grp * 512, &tm_kv,
                        256 * static_cast<int>(cta) + 128 * (pw >> 1), v[0], v[1], v[2], v[3], full, pol);
          if (lane == 0 && pw == 0) atomicMax(last_armed + slot, static_cast<int>(use));
          if (lane == 0 && pw == 0) MLA_TRACE_EVENT(1, g);
        }
      }
      ++g;
    }
    named_bar_sync(9, 32 * kProducers);
    if (pw == 0 && lane < kLatBlocks + kRopeSlots) {
      const int u = last_armed[lane];
      const int bfull = lane < kLatBlocks ? bLatFull + lane : bRopeFull + (lane - kLatBlocks);
      if (u >= 0) drain_wait(bar(bfull), u & 1);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------- QK issuer + rope-query loader
    // One thread; it blocks on its barriers (no polling), so the warps that
    // share its scheduler keep their issue slots.
    if (lane == 0) {
      const uint64_t dk = sdesc(base + kOffLat, 16, 1024);         // latent block 0, K-major (B of QK)
      const uint64_t dr = sdesc(base + kOffRope, 16, 256, kLayoutSw32);   // rope slot 0 (B of QK)
      const uint64_t dqr = sdesc(base + kOffQR, 16, 256, kLayoutSw32);    // rope query hi (A of QK)
      auto D = [](uint64_t d, uint32_t byte_off) -> uint64_t { return d + (byte_off >> 4); };
      uint32_t g = 0, nitem = 0;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const int b = item_w(it, 0), s = item_w(it, 1), e = item_w(it, 2);
        if (!item_ok(p, nnz, b, s, e)) continue;
        const int nt = (e - s + T - 1) / T;
        // the senders load this item's query parts once its previous item's last QK is done
        if (!mbar_wait(bar(bQFull), nitem & 1, wc)) break;
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t d_s = tmem + kTmS + (g & 1) * 64;
          const uint32_t blk = g % kLatBlocks, rs = g % kRopeSlots;
          if (g >= 2 && !mbar_wait(bar(bSFree + (g & 1)), ((g >> 1) - 1) & 1, wc)) { ok = false; break; }
          if (!mbar_wait(bar(bLatFull + blk), (g / kLatBlocks) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          MLA_TRACE_EVENT(2, g);
          const uint64_t bk = D(dk, blk * kLatBlock);
#pragma unroll
          for (int k = 0; k < 8; ++k) {           // 256 latent dims = 8 K-steps of 32; A (query hi, lo) from TMEM
            umma_ts_f8(d_s, tmem + kTmQHi + 8 * k, D(bk, (k >> 2) * kAtom + (k & 3) * 32), kIdescQK, k != 0 ? 1u : 0u);
            umma_ts_f8(d_s, tmem + kTmQLo + 8 * k, D(bk, (k >> 2) * kAtom + (k & 3) * 32), kIdescQKLo, 1u);
          }
          MLA_TRACE_EVENT(10, g);
          if (!mbar_wait(bar(bRopeFull + rs), (g / kRopeSlots) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          MLA_TRACE_EVENT(12, g);
          const uint64_t br = D(dr, rs * kRopeAtom);
          // this CTA's 32 rope dims: one K-step, query hi then lo
          umma_ss_f8(d_s, dqr, br, kIdescQK, 1u);
          umma_ss_f8(d_s, D(dqr, kQRPlane), br, kIdescQKLo, 1u);
          umma_commit(bar(bRopeEmpty + rs));
          umma_commit(bar(bSFull + (g & 1)));
          if (j == nt - 1) umma_commit(bar(bQEmpty));
          MLA_TRACE_EVENT(3, g);
        }
        ++nitem;
      }
      umma_commit(bar(bDrain));
      drain_wait(bar(bDrain), 0);
    }
    __syncwarp();
  } else if (warp == kLoaderWarp) {
    // ----------------------------------------------------------- PV issuer
    if (lane == 0) {
      const uint64_t dv = sdesc(base + kOffLat, kAtom, 1024);      // latent block 0, MN-major (B of PV)
      const uint64_t dp = sdesc(base + kOffX, 16, 1024);           // P in exchange slot 0 (A of PV)
      auto D = [](uint64_t d, uint32_t byte_off) -> uint64_t { return d + (byte_off >> 4); };
      const uint16_t peer_mask = static_cast<uint16_t>(1u << peer);
      uint32_t g = 0, nitem = 0;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const int b = item_w(it, 0), s = item_w(it, 1), e = item_w(it, 2);
        if (!item_ok(p, nnz, b, s, e)) continue;
        const int nt = (e - s + T - 1) / T;
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t xs = g % kXSlots, blk = g % kLatBlocks;
          if (!mbar_wait(bar(bPFull + xs), (g / kXSlots) & 1, wc)) { ok = false; break; }
          if (j == 0 && nitem > 0 && !mbar_wait(bar(bOEmpty), (nitem - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          MLA_TRACE_EVENT(4, g);
          const uint64_t bv = D(dv, blk * kLatBlock);
          const uint64_t ap = D(dp, xs * kXSlot);
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {        // 64 tokens = 2 K-steps of 32; P hi (bytes 0-63), lo (64-127)
            umma_ss_f8(tmem + kTmO, D(ap, ks * 32), D(bv, ks * 4096), kIdescPV, (j == 0 && ks == 0) ? 0u : 1u);
            umma_ss_f8(tmem + kTmO, D(ap, 64 + ks * 32), D(bv, ks * 4096), kIdescPV, 1u);
          }
          umma_commit(bar(bLatEmpty + blk));
          umma_commit_mc(bar(bXFree + xs), peer_mask);         // the peer may send into this slot again
          umma_commit(bar(bPvDone + (g & 1)));
          if (j == nt - 1) umma_commit(bar(bOFull));
          MLA_TRACE_EVENT(5, g);
        }
        ++nitem;
      }
      umma_commit(bar(bDrain));
      drain_wait(bar(bDrain), 0);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------- sender and softmax warps
    const bool is_sender = warp >= kSendWarp0;
    const int q = warp & 3, th = (warp >> 2) & 1;   // TMEM lane quadrant, token half of every tile
    const int h = 32 * q + lane;                 // head == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const bool head_ok = h < H;
    const uint32_t sw = static_cast<uint32_t>(h & 7);      // 16-byte chunk c of row h sits at c ^ (h mod 8)
    const uint32_t xrow_peer = mapa_shared(base + kOffX + h * 128, peer);
    const uint32_t xe_peer = mapa_shared(base + kOffXE + (th * 128 + h) * 4, peer);
    const uint32_t xlo_peer = mapa_shared(base + kOffXLo + h * 16, peer);
    const uint32_t xfull_peer = mapa_shared(bar(bXFull), peer);
    float* red_max = reinterpret_cast<float*>(smem + kOffRed);            // [2][2][128]
    float* red_l = red_max + 2 * 2 * 128;                                 // [2 halves][128]
    float m_ref = 0.f, l_sum = 0.f;
    float q_fac = 1.f;                           // 2^-a of this item's head scaling (senders and softmax)
    const float sl_kv = p.scale_log2 * kv_scale; // decoded partials in log2 units of the true scores
    auto wait = [&](uint32_t bb, uint32_t par, bool cluster_scope) {
      if (aborted) return;
      bool r = true;
      if (lane == 0) r = cluster_scope ? mbar_wait<true>(bb, par, wc) : mbar_wait(bb, par, wc);
      r = __shfl_sync(0xffffffffu, r, 0);
      if (!r) aborted = true;
    };

    // -- tile g of this CTA: quantise this warp's 32 partial scores of row h
    //    and push the codes to the peer (the softmax warps read the same
    //    partials from TMEM themselves)
    auto send = [&](uint32_t g) {
      const uint32_t sb = g & 1, xs = g % kXSlots;
      const uint32_t tm_s = tmem + lane_off + kTmS + sb * 64 + th * TH;
      wait(bar(bSFull + sb), (g >> 1) & 1, false);
      if (threadIdx.x == 32 * kSendWarp0) MLA_TRACE_EVENT(6, g);
      tc_fence_after();
      uint32_t qw[16], lb[16];
      int e_own;
      {
        uint32_t r[32];
        if (!aborted) {
          tmem_ld16(tm_s, *reinterpret_cast<uint32_t(*)[16]>(r));
          tmem_ld16(tm_s + 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16));
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(bSFree + sb));
        // this CTA's partial in the units both CTAs share: times 2^-a (exact)
        {
          const float2 qf2 = f2_pack(q_fac, q_fac);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 v = f2_mul(f2_pack(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), qf2);
            r[i] = __float_as_uint(v.x);
            r[i + 1] = __float_as_uint(v.y);
          }
        }
        // the step is 2^(e-21), e the exponent of max|s| nudged up by 2^-21 so
        // that no code rounds to 2^22
        float mx = 0.f;
#pragma unroll
        for (int i = 0; i < 32; i += 2) mx = max3(mx, fabsf(__uint_as_float(r[i])), fabsf(__uint_as_float(r[i + 1])));
        mx *= 1.000000476837158203125f;
        e_own = max(static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127, -100);
        const float inv = pow2i(min(21 - e_own, 127));
        const float2 inv2 = f2_pack(inv, inv), enc2 = f2_pack(kEncBias, kEncBias);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 t = f2_fma(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), inv2, enc2);
          qw[i] = __byte_perm(__float_as_uint(t.x), __float_as_uint(t.y), 0x6521);   // u >> 8, two codes
          lb[i] = __byte_perm(__float_as_uint(t.x), __float_as_uint(t.y), 0x0040);   // u & 255, two codes
        }
      }
      if (threadIdx.x == 32 * kSendWarp0) MLA_TRACE_EVENT(13, g);
      // push into the peer's slot xs once the peer's PV(g - kXSlots) has read it
      if (g >= kXSlots) wait(bar(bXFree + xs), ((g / kXSlots) - 1) & 1, true);
      if (threadIdx.x == 32 * kSendWarp0) MLA_TRACE_EVENT(14, g);
      if (!aborted) {
        const uint32_t fb = xfull_peer + 8u * xs;
        const uint32_t dst = xrow_peer + xs * kXSlot;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t c = static_cast<uint32_t>(4 * th + k);
          st_async_v4(dst + ((c ^ sw) << 4), qw[4 * k], qw[4 * k + 1], qw[4 * k + 2], qw[4 * k + 3], fb);
        }
        // low bytes: 32 codes of this row and half as 2 chunks of 16, chunk k
        // of half th at row h of block (2 th + k)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) w[i] = __byte_perm(lb[8 * k + 2 * i], lb[8 * k + 2 * i + 1], 0x5410);
          st_async_v4(xlo_peer + xs * kXLoSlot + static_cast<uint32_t>((2 * th + k) * 128) * 16u, w[0], w[1], w[2], w[3],
                      fb);
        }
        st_async_b32(xe_peer + xs * kXeSlot, static_cast<uint32_t>(e_own), fb);
      }
      if (threadIdx.x == 32 * kSendWarp0) MLA_TRACE_EVENT(8, g);
    };

    // -- tile g (j-th of an item of n tokens): add the peer's rows, softmax, P
    auto softmax = [&](uint32_t g, int j, int n) {
      const uint32_t sb = g & 1, xs = g % kXSlots;
      const uint32_t tm_s = tmem + lane_off + kTmS + sb * 64 + th * TH;
      // arm slot xs for the peer's rows of tile g: done here, by the warp that
      // also waits on it, so the arm for tile g + kXSlots cannot come before
      // this tile's phase has completed (the peer's bytes may land either side)
      if (warp == 0 && lane == 0 && !aborted) mbar_arrive_expect_tx(bar(bXFull + xs), kXBytes);
      wait(bar(bSFull + sb), (g >> 1) & 1, false);
      uint32_t sv[32];
      if (!aborted) {
        tc_fence_after();
        tmem_ld16(tm_s, *reinterpret_cast<uint32_t(*)[16]>(sv));
        tmem_ld16(tm_s + 16, *reinterpret_cast<uint32_t(*)[16]>(sv + 16));
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[i] = 0;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !aborted) mbar_arrive(bar(bSFree + sb));
      wait(bar(bXFull + xs), (g / kXSlots) & 1, true);
      if (threadIdx.x == 0) MLA_TRACE_EVENT(9, g);
      // s = (own exact partial x 2^-a + the peer's decoded one) in log2 units; -inf past the item end
      uint8_t* xrow = smem + kOffX + xs * kXSlot + h * 128;
      const int e_peer = !aborted ? *reinterpret_cast<const int*>(smem + kOffXE + xs * kXeSlot + (th * 128 + h) * 4)
                                  : -100;
      const float st_p = pow2i(max(e_peer - 21, -126));
      const float2 st2 = f2_pack(st_p, st_p), sth2 = f2_pack(256.f * st_p, 256.f * st_p);
      const float2 dec2 = f2_pack(-kDecHi * st_p, -kDecHi * st_p);
      const float2 sl2 = f2_pack(sl_kv, sl_kv), qf2 = f2_pack(q_fac, q_fac);
#pragma unroll
      for (int k = 0; k < 4; ++k) {            // 8 tokens per 16-byte chunk
        const uint32_t c = static_cast<uint32_t>(4 * th + k);
        uint4 pv = make_uint4(0x40004000u, 0x40004000u, 0x40004000u, 0x40004000u);   // code of 0 (u = 2^22)
        uint4 lv = make_uint4(0, 0, 0, 0);
        if (!aborted) {
          pv = *reinterpret_cast<const uint4*>(xrow + ((c ^ sw) << 4));
          // low bytes of tokens 8k..8k+7 of this half: bytes 8 (k & 1) .. of chunk (2 th + k / 2)
          lv = *reinterpret_cast<const uint4*>(smem + kOffXLo + xs * kXLoSlot + ((2 * th + (k >> 1)) * 128 + h) * 16);
        }
        const uint32_t pq[4] = {pv.x, pv.y, pv.z, pv.w};
        const uint32_t lw[2] = {(k & 1) ? lv.z : lv.x, (k & 1) ? lv.w : lv.y};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = 8 * k + 2 * i;
          const float2 f = f2_pack(__uint_as_float(__byte_perm(pq[i], 0x4B000000u, 0x7610)),
                                   __uint_as_float(__byte_perm(pq[i], 0x4B000000u, 0x7632)));
          const uint32_t lo2 = lw[i >> 1] >> (16 * (i & 1));     // the two low bytes of tokens t, t + 1
          const float2 fl = f2_pack(__uint_as_float(__byte_perm(lo2, 0x4B000000u, 0x7660)),
                                    __uint_as_float(__byte_perm(lo2, 0x4B000000u, 0x7661)));
          const float2 sp = f2_fma(fl, st2, f2_fma(f, sth2, dec2));
          const float2 s2 = f2_mul(f2_fma(f2_pack(__uint_as_float(sv[t]), __uint_as_float(sv[t + 1])), qf2, sp), sl2);
          sv[t] = __float_as_uint(s2.x);
          sv[t + 1] = __float_as_uint(s2.y);
        }
      }
      const int nvalid = n - j * T - th * TH;
      if (nvalid < TH) {
#pragma unroll
        for (int t = 0; t < TH; ++t)
          if (t >= nvalid) sv[t] = __float_as_uint(-INFINITY);
      }
      // the half row's maximum as a tree (short dependency chains)
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        mx8[i] = max3(__uint_as_float(sv[4 * i]), __uint_as_float(sv[4 * i + 1]),
                      fmaxf(__uint_as_float(sv[4 * i + 2]), __uint_as_float(sv[4 * i + 3])));
      const float mh = fmaxf(max3(mx8[0], mx8[1], mx8[2]), max3(max3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
      // row maximum over the tile: combine with the partner warp (other token half)
      float* rm = red_max + (g & 1) * 256;
      rm[th * 128 + h] = mh;
      named_bar_sync(1 + q, 64);
      const float mt = fmaxf(rm[h], rm[128 + h]);
      if (j == 0 || m_ref == -INFINITY) {
        // an item's first tile sets the reference; so does the first tile
        // with a valid score when a causal query row had none before (O and
        // the row sum are still zero then)
        m_ref = mt;
        if (j == 0) l_sum = 0.f;
      } else {
        const bool need = mt > m_ref + 3.f;   // P' <= 2^8 (see below)
        if (__any_sync(0xffffffffu, need)) {
          // rescale this warp's half of O (128 columns) after the previous PV has
          // landed.  PV(g-3) is complete here (the peer sent tile g only after
          // this CTA's PV(g - kXSlots) had freed slot g mod kXSlots, and
          // kXSlots <= 3), so the barrier of tile g-1 cannot be a lap behind.
          wait(bar(bPvDone + ((g - 1) & 1)), ((g - 1) >> 1) & 1, false);
          tc_fence_after();
          const float alpha = need ? ex2_approx(m_ref - mt) : 1.f;
          if (need) {
            m_ref = mt;
            l_sum *= alpha;
          }
          if (!aborted) {
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              uint32_t o[16];
              const uint32_t ta = tmem + lane_off + kTmO + 128 * th + 16 * c;
              tmem_ld16(ta, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st16(ta, o);
            }
            tmem_wait_st();
          }
          tc_fence_before();
        }
      }
      // P = 2^(s - m_ref) as E4M3 hi and lo, written over the peer's rows
      // (K-major, 128-byte swizzle): token t of the tile is byte t (hi) and
      // byte 64 + t (lo) of row h; this warp's 32 tokens are two 16-byte
      // chunks of each part
      // P' = 2^(s - m_ref + 5): the reference moves once a tile's maximum is
      // more than 3 above it, so P' <= 256 and the row maximum's weight is at
      // least 32; lo (unscaled: it shares the accumulator with hi) is exact
      // to E4M3's precision down to weights 2^-7 of that and within 2^-10
      // below, which stays under 2^-9 of the output even over thousands of
      // such tokens; lse takes the 2^5 out
      const float m_eff = m_ref == -INFINITY ? 0.f : m_ref;   // a row with no valid score yet: P = 0
      const float2 nm2 = f2_pack(5.f - m_eff, 5.f - m_eff);
      float2 l4[4] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f), f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
      for (int k = 0; k < 2; ++k) {              // 16 tokens per chunk
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = 16 * k + 2 * i;
          const float2 d = f2_add(f2_pack(__uint_as_float(sv[t]), __uint_as_float(sv[t + 1])), nm2);
          const float a = ex2_approx(d.x), e2 = ex2_approx(d.y);
          uint32_t h2, l2;
          e4m3x2_split(a, e2, h2, l2);
          l4[i & 3] = f2_add(l4[i & 3], f2_pack(a, e2));   // four independent sums (fp32 P, as the bf16 kernel)
          if (i & 1) {
            ph[i >> 1] |= h2 << 16;
            pl[i >> 1] |= l2 << 16;
          } else {
            ph[i >> 1] = h2;
            pl[i >> 1] = l2;
          }
        }
        const uint32_t ch = static_cast<uint32_t>(2 * th + k), cl = static_cast<uint32_t>(4 + 2 * th + k);
        if (!aborted) {
          *reinterpret_cast<uint4*>(xrow + ((ch ^ sw) << 4)) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
          *reinterpret_cast<uint4*>(xrow + ((cl ^ sw) << 4)) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
        }
      }
      const float2 l2 = f2_add(f2_add(l4[0], l4[1]), f2_add(l4[2], l4[3]));
      l_sum += l2.x + l2.y;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && !aborted) mbar_arrive(bar(bPFull + xs));
      if (threadIdx.x == 0) MLA_TRACE_EVENT(7, g);
    };

    // -- after an item's last tile: 1/l, O (this warp's 128 columns) and lse
    auto epilogue = [&](int b, int part, uint32_t nitem) {
      if (threadIdx.x == 0 && nitem < 24) MLA_TRACE_RAW(15, 8 + 2 * nitem, clock64());
      // the row sum over the tile halves, added in the same order by both warps
      red_l[th * 128 + h] = l_sum;
      named_bar_sync(1 + q, 64);
      const float lsum = red_l[h] + red_l[128 + h];
      wait(bar(bOFull), nitem & 1, false);
      tc_fence_after();
      const bool part_ok = part < p.max_partials;   // a device-only plan naming a partial past the workspace
      if (!part_ok && threadIdx.x == 0) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
      if (!aborted && part_ok) {
        const float inv = lsum > 0.f ? kv_scale / lsum : 0.f;   // no valid score: out = 0
        // rows of this warp's lane group (4 lanes): after the block transpose
        // lane i of group m holds columns 8i..8i+7 (fp32) of rows 4m..4m+3 of
        // the warp's 32, so each store instruction writes whole 128-byte lines
        const int h4 = 32 * q + 4 * (lane >> 2), bi = lane & 3;
        const size_t col0 = 256 * static_cast<size_t>(cta) + 128 * th;
        const size_t row0 = part < 0 ? static_cast<size_t>(b) * H : static_cast<size_t>(part) * H;
        float* dst_f = nullptr;
        __nv_bfloat16* dst_h = nullptr;
        if (part >= 0) dst_f = p.part_o + row0 * kLatent + col0;
        else if (p.out_bf16) dst_h = reinterpret_cast<__nv_bfloat16*>(p.out) + row0 * kLatent + col0;
        else dst_f = reinterpret_cast<float*>(p.out) + row0 * kLatent + col0;
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {          // 32 columns per TMEM round trip
          uint32_t o[32];
          {
            uint32_t a[16], c[16];
            tmem_ld16(tmem + lane_off + kTmO + 128 * th + 32 * cb, a);
            tmem_ld16(tmem + lane_off + kTmO + 128 * th + 32 * cb + 16, c);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) { o[i] = a[i]; o[16 + i] = c[i]; }
          }
          if (dst_f) {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * inv);
            transpose4_blocks<8>(o, lane);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint32_t v[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] = o[8 * k + e];
              if (h4 + k < H) st_global_v8(dst_f + static_cast<size_t>(h4 + k) * kLatent + 32 * cb + 8 * bi, v);
            }
          } else {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
            transpose4_blocks<4>(w, lane);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (h4 + k < H)
                st_global_v4(dst_h + static_cast<size_t>(h4 + k) * kLatent + 32 * cb + 8 * bi, w[4 * k], w[4 * k + 1],
                             w[4 * k + 2], w[4 * k + 3]);
          }
        }
        if (cta == 0 && th == 0 && head_ok) {
          const float l = lsum > 0.f ? (m_ref + __log2f(lsum) - 5.f) * 0.69314718055994531f : -INFINITY;
          if (part < 0) { if (p.lse) p.lse[static_cast<size_t>(b) * H + h] = l; }
          else p.part_lse[static_cast<size_t>(part) * H + h] = l;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !aborted) mbar_arrive(bar(bOEmpty));
      if (threadIdx.x == 0 && nitem < 24) MLA_TRACE_RAW(15, 9 + 2 * nitem, clock64());
    };

    // the head's scale a: max |q 2^a| over this CTA's 256 latent + 32 rope
    // dims in [128, 256).  Senders and softmax warps each compute it from the
    // query, with the same code, so both hold the same 2^-a.
    auto head_exp = [&](int b) -> int {
      const uint4* qn = reinterpret_cast<const uint4*>(p.q_nope + (static_cast<size_t>(b) * H + h) * kLatent + 256 * cta);
      const uint4* qr = reinterpret_cast<const uint4*>(p.q_rope + (static_cast<size_t>(b) * H + h) * kRope + 32 * cta);
      auto absmax8 = [](const uint4& v, float m) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
        return m;
      };
      float amax = 0.f;
      if (head_ok) {
#pragma unroll 4
        for (int i = 0; i < 32; ++i) amax = absmax8(__ldg(qn + i), amax);
#pragma unroll
        for (int i = 0; i < 4; ++i) amax = absmax8(__ldg(qr + i), amax);
      }
      int a = 0;
      if (amax > 0.f && amax <= 3.0e38f) {
        int e;
        frexpf(amax, &e);
        a = min(126, max(-126, 8 - e));
      }
      return a;
    };

    uint32_t g = 0, nitem = 0;
    for (int it = it0; it < it1; ++it) {
      const int b = item_w(it, 0), s = item_w(it, 1), e = item_w(it, 2);
      const int part = item_w(it, 3);
      if (!item_ok(p, nnz, b, s, e)) continue;
      const int n = e - s, nt = (n + T - 1) / T;
      if (is_sender) {
        // -- this item's query parts: the head's scale a from this CTA's 256
        //    latent + 32 rope dims (read before the wait for the previous item's
        //    last QK: an item's first QK waits on this work), then, after that
        //    wait, this warp's 128 latent dims as hi / lo into TMEM and
        //    (token-half-0 warps) the 32 rope dims as hi / lo into shared memory
        const int a = !aborted ? head_exp(b) : 0;
        if (nitem > 0) wait(bar(bQEmpty), (nitem - 1) & 1, false);
        tc_fence_after();
        if (!aborted) {
          const uint4* qn = reinterpret_cast<const uint4*>(p.q_nope + (static_cast<size_t>(b) * H + h) * kLatent +
                                                           256 * cta);
          const uint4* qr = reinterpret_cast<const uint4*>(p.q_rope + (static_cast<size_t>(b) * H + h) * kRope +
                                                           32 * cta);
          q_fac = ldexpf(1.f, -a);
          const float up = ldexpf(1.f, a);
          // 8 bf16 -> 2 words of E4M3 hi and 2 of E5M2 lo
          auto split8 = [&](const uint4& v, uint32_t& h0, uint32_t& h1, uint32_t& l0, uint32_t& l1) {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t hh[4], ll[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float u0 = __uint_as_float(w[i] << 16) * up, u1 = __uint_as_float(w[i] & 0xFFFF0000u) * up;
              hh[i] = e4m3x2(u0, u1);
              const float2 hv = e4m3x2_value(hh[i]);
              ll[i] = e5m2x2(u0 - hv.x, u1 - hv.y);   // the difference is exact in fp32
            }
            h0 = hh[0] | (hh[1] << 16);
            h1 = hh[2] | (hh[3] << 16);
            l0 = ll[0] | (ll[1] << 16);
            l1 = ll[2] | (ll[3] << 16);
          };
#pragma unroll
          for (int c = 0; c < 2; ++c) {            // this warp's 128 dims: 2 x 16 columns of each part
            uint32_t rh[16], rl[16];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint4 v = head_ok ? __ldg(qn + 16 * th + 8 * c + k) : make_uint4(0, 0, 0, 0);
              split8(v, rh[2 * k], rh[2 * k + 1], rl[2 * k], rl[2 * k + 1]);
            }
            tmem_st16(tmem + lane_off + kTmQHi + 32 * th + 16 * c, rh);
            tmem_st16(tmem + lane_off + kTmQLo + 32 * th + 16 * c, rl);
          }
          tmem_wait_st();
          if (th == 0) {
            // rope query row h: 32 dims = two 16-byte chunks per part (32-byte swizzle)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t h4[4], l4[4];
              const uint4 v0 = head_ok ? __ldg(qr + 2 * c) : make_uint4(0, 0, 0, 0);
              const uint4 v1 = head_ok ? __ldg(qr + 2 * c + 1) : make_uint4(0, 0, 0, 0);
              split8(v0, h4[0], h4[1], l4[0], l4[1]);
              split8(v1, h4[2], h4[3], l4[2], l4[3]);
              const uint32_t off = (h >> 3) * 256 + (h & 7) * 32 + (((c ^ (h >> 2)) & 1) << 4);
              *reinterpret_cast<uint4*>(smem + kOffQR + off) = make_uint4(h4[0], h4[1], h4[2], h4[3]);
              *reinterpret_cast<uint4*>(smem + kOffQR + kQRPlane + off) = make_uint4(l4[0], l4[1], l4[2], l4[3]);
            }
            fence_proxy_async_smem();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(bQFull));
        for (int j = 0; j < nt; ++j, ++g) send(g);
      } else {
        // multi-query: row h is query h / (H / q_len) of its request, which
        // sees the first L - q_len + 1 + i rows of the request's context
        int n_row = n;
        if (p.q_len > 1) {
          const int lo = __ldg(p.kv_indptr + b), hi = __ldg(p.kv_indptr + b + 1);
          const int i = h / (H / p.q_len);
          n_row = max(0, min(n, (hi - lo) - p.q_len + 1 + i - (s - lo)));
        }
        q_fac = ldexpf(1.f, -head_exp(b));
        for (int j = 0; j < nt; ++j, ++g) softmax(g, j, n_row);
        epilogue(b, part, nitem);
      }
      ++nitem;
    }
  }

  // A CTA that gave up may still have the peer's rows in flight towards it.
  const bool gave_up = __syncthreads_or(aborted) != 0;
  tc_fence_before();
  cluster_sync_all();                            // no CTA leaves while its peer may still write to it
  tc_fence_after();
  if (gave_up && threadIdx.x == 0) {
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 50000ull) {
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    MLA_TRACE_RAW(15, 1, static_cast<long long>(globaltimer()));
    MLA_TRACE_RAW(15, 4, clock64());
  }
  if (warp == kLoaderWarp) tmem_dealloc(tmem, 512);
}

}  // namespace pair8

int launch_pair8(int heads, const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const DecodeParams& p,
                 float kv_scale, int workers, cudaStream_t stream) {
  if (heads < 48 || heads > 128 || heads % 16 != 0) return MLA_ERR_UNSUPPORTED;
  if (!set_smem_limit(reinterpret_cast<const void*>(&pair8::pair8_kernel), pair8::kSmemBytes)) return MLA_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * workers, 1, 1);
  cfg.blockDim = dim3(pair8::kThreads, 1, 1);
  cfg.dynamicSmemBytes = pair8::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // the prologue overlaps the previous kernel
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, pair8::pair8_kernel, tm_lat, tm_rope, p, kv_scale) != cudaSuccess) return MLA_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace mla
