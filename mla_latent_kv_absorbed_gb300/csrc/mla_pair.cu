// Absorbed MLA decode for many heads (H = 48..128, step 16) on sm_103a.
//
// With 128 query heads the heads fill the tensor core's 128-row M side, but
// one SM cannot hold the whole problem: the fp32 output O[128 heads x 512]
// alone is all 512 TMEM columns.  So a worker is a cluster of two CTAs that
// split the latent dimensions: CTA c owns latent dims D_c = [256c, 256c+256)
// of every row and half of the rope key, and the softmax of half the heads.
//
//   QK (per CTA, partial):  S_c[128 h x 64 tok] = Q[:, D_c] . K[:, D_c]^T  (+ its rope half)
//   exchange 1:             each CTA sends its fp32 partial of the PEER's heads
//                           to the peer (distributed shared memory)
//   softmax (own heads):    s = S_c + S_peer, an fp32 sum of the two halves,
//                           online softmax, P as bf16
//   exchange 2:             each CTA copies its heads' P rows to the peer
//   PV (per CTA):           O_c[128 h x 256] += P[128 x 64 tok] . V[64 tok x D_c]
//
// so no product is computed twice, no latent byte is loaded twice, and no
// score is held in less than fp32 on the way.  ("实现差距：MLA 与 DeepSeek V3",
// section 2.4: the latent and rope dot products are summed and scaled by
// sm_scale, FA2-style online softmax, the latent rows reused as the values;
// "Attention backends", paragraph "MLA": every KV byte used by all 128 heads.)
//
// The exchange is the narrow path: an SM moves only about 9 bytes per cycle
// to its cluster peer.  Per 64-token tile each CTA sends 64 heads x 64
// partial scores x 4 B (16 KB) and 64 rows x 128 B of P (8 KB); the softmax
// of a head runs in one CTA only, so neither it nor the scores are
// duplicated.
//
// Rows.  In CTA c, TMEM lane / P row / O row r < H/2 is this CTA's head
// c*H/2 + r ("own"), and row 64 + r is the peer's head (1-c)*H/2 + r; other
// rows are padding (zero query).  Own rows sit in lane quadrants 0-1, peer
// rows in quadrants 2-3, so the warps of quadrants 0-1 take the softmax and
// those of quadrants 2-3 the exchange of the peer's rows.
//
// TMEM (512 columns per CTA): O_c [0,256) fp32; the query's latent half
// [256,384) as packed bf16 (A operand of QK); two score buffers [384,448),
// [448,512) holding this CTA's raw fp32 partial.
//
// Shared memory per CTA: a ring of 4 latent blocks (64 tokens x 256 dims,
// 32 KB, TMA gather4), 4 rope atoms (4 KB: this CTA's 32 rope dims, 64-byte
// swizzle), the rope query (8 KB), 2 P slots (128 rows x 64 tokens bf16, the
// A operand of PV: rows 0-63 written here, rows 64-127 copied in by the
// peer), 2 receive slots (the peer's fp32 partials of this CTA's heads,
// 16 KB), 2 side slots (the peer's rescale factors and row sums), reduction
// buffers.
//
// Warp roles per CTA (800 threads).  Row warp w < 16 sits on lane quadrant
// w & 3 and takes tokens 16(w >> 2)..+15 of every tile and latent columns
// 64(w >> 2)..+63 of O:
//   quadrants 0-1 (own rows)  softmax: add the peer's partial, row maximum
//               over the four warps of the quadrant, lazy reference, P, row
//               sums; rescale and write out their rows of O
//   quadrants 2-3 (peer rows) pushers: push this CTA's partial of the peer's
//               rows (st.async); write those rows of O out after an item
//   warp 16     QK issuer and rope-query loader (one thread)
//   warp 17     TMEM allocator and PV issuer (one thread), which also copies
//               this CTA's P rows to the peer (bulk copy)
//   warps 18-19 takers (lane quadrants 2, 3): once the peer's P rows of a
//               tile have landed, apply its rescale factors to the peer's
//               rows of O, then release the tile's PV.  Kept apart from the
//               pushers so that no push ever waits for a P exchange.
//   warps 20-24 gather producers: latent atoms 0-3 of the CTA's half, rope
//
// Per tile g (S buffer, receive slot and P slot g mod 2): QK(g) -> pushers
// push the peer's rows, softmax warps read their own rows (freeing the S
// buffer for QK(g+2)) -> the peer's partials land -> softmax, own P rows ->
// the PV issuer copies them to the peer -> the peer's P rows land, the
// takers apply the peer's rescale factors -> PV(g), which frees the latent
// block and P slot g mod 2.  An item's output is written after the next
// item's first tile has been pushed and taken through its softmax.
//
// The reference maximum moves lazily: only when a tile's maximum exceeds it
// by more than 64 (log2 units), so O is rescaled rarely.  P stays below 2^64
// and O, l below 2^100, well inside fp32; a score more than 126 below the
// reference flushes to zero, at less than 2^-126 of the largest weight.
#include "mla_device.cuh"
#include "mla_launch.h"

namespace mla {
namespace pair {

constexpr int T = 64;                        // tokens per tile
constexpr int kGroup = 16;                   // tokens of a tile per row warp
constexpr int kRowWarps = 16;                // warps 0-15
constexpr int kOwnWarps = 8;                 // the row warps of quadrants 0-1
constexpr int kMmaWarp = 16, kPvWarp = 17;
constexpr int kTakeWarp0 = 18, kTakeWarps = 2;   // lane quadrants 2 and 3: the peer's rows of O
constexpr int kProducerWarp0 = kTakeWarp0 + kTakeWarps;
constexpr int kProducers = 5;                // latent atoms 0-3 and the rope
constexpr int kCopyWarp = kProducerWarp0 + kProducers;   // copies this CTA's P rows to the peer
constexpr int kThreads = 32 * (kCopyWarp + 1);
constexpr int kLatBlocks = 4;                // ring of latent blocks
constexpr int kRopeSlots = 4;
constexpr int kLead = 3;                     // a producer issues tile g once tile g - kLead has landed
constexpr int kXSlots = 2;                   // receive slots
constexpr int kPSlots = 2;                   // P slots (also the parity of "PV(g) done")
constexpr int kAtom = T * 128;               // 8 KB: 64 tokens x 64 dims
constexpr int kLatBlock = 4 * kAtom;         // 32 KB: 64 tokens x 256 dims
constexpr int kRopeAtom = T * 64;            // 4 KB: 64 tokens x this CTA's 32 rope dims (64-byte swizzle)
constexpr int kQRBytes = 128 * 64;           // rope query: 128 rows x this CTA's 32 rope dims
constexpr int kPSlot = 128 * 128;            // 128 rows x 64 tokens bf16 (K-major, 128-byte swizzle)
constexpr int kXSlot = 64 * T * 4;           // 64 own rows x 64 tokens fp32 (256-byte rows)
constexpr int kSideSlot = 2 * 64 * 4;        // [64] rescale factors, [64] row sums
constexpr int kOffLat = 0;
constexpr int kOffRope = kOffLat + kLatBlocks * kLatBlock;
constexpr int kOffQR = kOffRope + kRopeSlots * kRopeAtom;
constexpr int kOffP = kOffQR + kQRBytes;
constexpr int kOffX = kOffP + kPSlots * kPSlot;
constexpr int kOffSide = kOffX + kXSlots * kXSlot;              // the peer's rescale factors / row sums
constexpr int kOffSideOut = kOffSide + kPSlots * kSideSlot;     // this CTA's, copied to the peer with P
constexpr int kOffRed = kOffSideOut + kPSlots * kSideSlot;   // [2][4][64] tile maxima, [4][64] row sums
constexpr int kOffLPeer = kOffRed + (2 * 4 * 64 + 4 * 64) * 4;   // [2 items][64] the peer's row sums, kept by the takers
constexpr int kOffBar = kOffLPeer + 2 * 64 * 4;
// barriers
constexpr int bLatFull = 0;
constexpr int bLatEmpty = bLatFull + kLatBlocks;
constexpr int bRopeFull = bLatEmpty + kLatBlocks;
constexpr int bRopeEmpty = bRopeFull + kRopeSlots;
constexpr int bQFull = bRopeEmpty + kRopeSlots;
constexpr int bQEmpty = bQFull + 1;
constexpr int bSFull = bQEmpty + 1;          // [2] this CTA's partial is in the S buffer
constexpr int bSFree = bSFull + 2;           // [2] every row warp has read the S buffer
constexpr int bXFull = bSFree + 2;           // [kXSlots] the peer's partials have landed here
constexpr int bXFree = bXFull + kXSlots;     // [kXSlots] the PEER's receive slot may take this CTA's next partials
constexpr int bPFull = bXFree + kXSlots;     // [kPSlots] the own P rows are written
constexpr int bPeerP = bPFull + kPSlots;     // [kPSlots] the peer's P rows and side values have landed here
constexpr int bPeerOK = bPeerP + kPSlots;    // [kPSlots] the senders have applied the peer's rescale factors
constexpr int bPSlotMine = bPeerOK + kPSlots;   // [kPSlots] this CTA's PV of the slot's tile is done
constexpr int bPSlotPeer = bPSlotMine + kPSlots;  // [kPSlots] the PEER's PV of the slot's tile is done
constexpr int bOFull = bPSlotPeer + kPSlots;
constexpr int bOEmpty = bOFull + 1;
constexpr int bDrain = bOEmpty + 1;
constexpr int kNumBars = bDrain + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffLast = kOffMisc + 16;      // [kLatBlocks + kRopeSlots] last armed use
constexpr int kSmemBytes = kOffLast + 4 * (kLatBlocks + kRopeSlots) + 1024;
constexpr int kTmO = 0, kTmQ = 256, kTmS = 384;
constexpr uint32_t kIdescQK = idesc_bf16(128, T, false, false);     // M=128 rows, N=64 tokens
constexpr uint32_t kIdescPV = idesc_bf16(128, 256, false, true);    // N=256 dims, B (V) MN-major
static_assert(kProducers == 5, "producers 0-3 gather the latent atoms, producer 4 the rope");
static_assert(kThreads == 832, "26 warps (registers are budgeted as for 28)");
static_assert(kTakeWarp0 % 4 == 2, "the taker warps sit on lane quadrants 2 and 3");
static_assert(kLead < kLatBlocks && kLead <= kRopeSlots, "a ring slot's phase must not be lapped while waited on");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffRope % 1024 == 0 && kOffQR % 1024 == 0 && kOffP % 1024 == 0 && kOffX % 1024 == 0 &&
                  kOffSide % 16 == 0 && kOffBar % 8 == 0,
              "alignment");
static_assert(kPSlots == 2, "bPSlotMine doubles as the 'PV(g) done' barrier of parity g mod 2");

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

// Head of row r in CTA `cta` for H = 2 Hh heads, or -1 for a padding row.
__device__ __forceinline__ int row_head(int r, uint32_t cta, int Hh) {
  if (r < 64) return r < Hh ? static_cast<int>(cta) * Hh + r : -1;
  return r - 64 < Hh ? static_cast<int>(cta ^ 1u) * Hh + (r - 64) : -1;
}

__global__ void __launch_bounds__(kThreads, 1)
    pair_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_kr,
                const __grid_constant__ CUtensorMap tm_qr,
                const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t cta = cluster_ctarank();        // 0 or 1: which latent half, which heads
  const uint32_t peer = cta ^ 1u;
  auto bar = [&](int i) -> uint32_t { return base + kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* last_armed = reinterpret_cast<int*>(smem + kOffLast);
  const WaitCtx wc{abort_flag, p.status};
#ifdef MLA_TRACE
  if (threadIdx.x == 0) {
    MLA_TRACE_RAW(15, 0, static_cast<long long>(globaltimer()));
    MLA_TRACE_RAW(15, 3, clock64());
  }
#endif

  const int w = blockIdx.x >> 1;
  int it0, it1;
  plan_items(p, w, it0, it1);
  const int32_t* items = p.plan + p.items_off;
  const int H = p.heads, Hh = H >> 1;
  const int nnz = __ldg(p.kv_indptr + p.batch);   // loaded alongside the plan words

  if (threadIdx.x == 0) {
    for (int i = 0; i < kLatBlocks; ++i) { mbar_init(bar(bLatFull + i), 1); mbar_init(bar(bLatEmpty + i), 1); }
    for (int i = 0; i < kRopeSlots; ++i) { mbar_init(bar(bRopeFull + i), 1); mbar_init(bar(bRopeEmpty + i), 1); }
    mbar_init(bar(bQFull), kRowWarps + 1);       // the row warps (latent half) + the rope TMA
    mbar_init(bar(bQEmpty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bSFull + i), 1);
      mbar_init(bar(bSFree + i), kRowWarps);
    }
    for (int i = 0; i < kXSlots; ++i) {
      mbar_init(bar(bXFull + i), 1);             // own expect_tx; the bytes come from the peer
      mbar_init(bar(bXFree + i), 1);             // the peer's PV issuer (commit)
    }
    for (int i = 0; i < kPSlots; ++i) {
      mbar_init(bar(bPFull + i), kOwnWarps);
      mbar_init(bar(bPeerP + i), 1);             // own expect_tx; the bytes come from the peer
      mbar_init(bar(bPeerOK + i), kTakeWarps);
      mbar_init(bar(bPSlotMine + i), 1);         // this CTA's PV commit
      mbar_init(bar(bPSlotPeer + i), 1);         // the peer's PV commit
    }
    mbar_init(bar(bOFull), 1);
    mbar_init(bar(bOEmpty), kRowWarps);
    mbar_init(bar(bDrain), 2);                   // both issuers' final commits
    for (int i = 0; i < kLatBlocks + kRopeSlots; ++i) last_armed[i] = -1;
    *abort_flag = 0;
    fence_mbar_init();
  }
  // rope-query rows of padding heads stay zero (each TMA box has H/2 rows)
  for (int i = threadIdx.x; i < kQRBytes / 16; i += blockDim.x)
    *reinterpret_cast<uint4*>(smem + kOffQR + 16 * i) = make_uint4(0, 0, 0, 0);
  if (warp == kPvWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  cluster_sync_all();                            // both CTAs' barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the merge kernel may be launched now: it waits for this grid to finish
  griddep_launch_dependents();
  bool aborted = false;                          // set by the row and taker warps only

  if (warp >= kProducerWarp0 && warp < kCopyWarp) {
    // ------------------------------------------------------ gather producers
    // A warp completes one gather4 only every ~70-110 cycles, so a tile's
    // landing time is set by how many gathers one warp issues for it.  The
    // five producers split every tile evenly: producer pw < 4 gathers latent
    // atom pw of the CTA's half, producer 4 the rope atom; 16 gathers each.
    // Each loads its tile's slot numbers (lane l < 16: tokens 4l..4l+3)
    // before it waits for ring space; an out-of-range slot reads row 0 and
    // sets MLA_ERR_INDEX_OOB, the ragged tail repeats the last valid slot.
    const int pw = warp - kProducerWarp0;
    if (lane == 0 && pw == 0) tma_prefetch_desc(&tm_kv);
    if (lane == 0 && pw == 4) tma_prefetch_desc(&tm_kr);
    const uint64_t pol = l2_policy_evict_first();
    int it = it0, s = 0, n = 0;
    auto next_item = [&]() {                     // first usable item from `it` on
      for (; it < it1; ++it) {
        const int b = items[4 * it], s0 = items[4 * it + 1], e = items[4 * it + 2];
        if (item_ok(p, nnz, b, s0, e)) {
          if (pw == 0 && lane == 0 && !item_in_request(p, b, s0, e)) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
          s = s0;
          n = e - s0;
          return;
        }
        if (lane == 0 && pw == 0) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
      }
    };
    auto load_slots = [&](int t0, int (&v)[4]) {
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = __ldg(p.kv_indices + s + min(t0 + 4 * (lane & 15) + k, n - 1));
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
      if (oob && pw == 0) record_status(p.status, MLA_ERR_INDEX_OOB);
      // advance the cursor and prefetch the next tile's slot numbers
      t0 += T;
      if (t0 >= n) {
        ++it;
        next_item();
        t0 = 0;
      }
      if (it < it1) load_slots(t0, vn);
      {
        const bool rope = pw == 4;
        const uint32_t nslots = rope ? kRopeSlots : kLatBlocks;
        const uint32_t slot = g % nslots, use = g / nslots;
        const uint32_t full = bar((rope ? bRopeFull : bLatFull) + slot);
        bool e_ok = true;
        if (lane == 0 && use > 0) e_ok = mbar_wait(bar((rope ? bRopeEmpty : bLatEmpty) + slot), (use - 1) & 1, wc);
        if (lane == 0 && e_ok && g >= static_cast<uint32_t>(kLead)) {   // pace: tile g - kLead has landed
          const uint32_t gp = g - kLead;
          e_ok = mbar_wait(bar((rope ? bRopeFull : bLatFull) + gp % nslots), (gp / nslots) & 1, wc);
        }
        e_ok = __shfl_sync(0xffffffffu, e_ok, 0);
        if (!e_ok) { ok = false; break; }
        if (rope) {
          if (lane == 0) mbar_arrive_expect_tx(full, kRopeAtom);
          __syncwarp();
          if (lane < 16)
            tma_gather4(base + kOffRope + slot * kRopeAtom + lane * 256, &tm_kr, 512 + 32 * static_cast<int>(cta),
                        v[0], v[1], v[2], v[3], full, pol);
          if (lane == 0) atomicMax(last_armed + kLatBlocks + slot, static_cast<int>(use));
        } else {
          if (lane == 0 && pw == 0) mbar_arrive_expect_tx(full, kLatBlock);
          __syncwarp();
          if (lane < 16)
            tma_gather4(base + kOffLat + slot * kLatBlock + pw * kAtom + lane * 512, &tm_kv,
                        64 * (4 * static_cast<int>(cta) + pw), v[0], v[1], v[2], v[3], full, pol);
          if (lane == 0 && pw == 0) atomicMax(last_armed + slot, static_cast<int>(use));
          if (lane == 0 && pw == 0) MLA_TRACE_EVENT(0, g);
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
  } else if (warp == kCopyWarp) {
    // ------------------------------------------------------------- P copier
    // Tile g: once the softmax warps have written their P rows (so they have
    // also consumed the peer's partials of tile g), let the peer's pushers
    // refill that receive slot, and once the peer's PV of tile g - kPSlots
    // has freed the peer's P slot, copy the P rows and the side slot there.
    if (lane == 0) {
      // this CTA's rows 0..H/2-1 of a P slot are the peer's rows 64..64+H/2-1
      const uint32_t peer_p = mapa_shared(base + kOffP + 64 * 128, peer);
      const uint32_t peer_pbar = mapa_shared(bar(bPeerP), peer);
      const uint32_t peer_side = mapa_shared(base + kOffSide, peer);
      const uint32_t p_bytes = static_cast<uint32_t>(Hh) * 128u;
      const uint16_t peer_mask = static_cast<uint16_t>(1u << peer);
      uint32_t g = 0;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
        if (!item_ok(p, nnz, b, s, e)) continue;
        const int nt = (e - s + T - 1) / T;
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t ps = g % kPSlots, use = g / kPSlots;
          if (!mbar_wait(bar(bPFull + ps), use & 1, wc)) { ok = false; break; }
          // the arrive on the peer's barrier rides on a tensor-core commit: it
          // tracks no MMA of this thread, and unlike a thread's remote arrive
          // it does not queue behind the pushers' stores
          umma_commit_mc(bar(bXFree + g % kXSlots), peer_mask);
          if (g >= static_cast<uint32_t>(kPSlots) && !mbar_wait<true>(bar(bPSlotPeer + ps), (use - 1) & 1, wc)) {
            ok = false;
            break;
          }
          bulk_copy_to_peer(peer_p + ps * kPSlot, base + kOffP + ps * kPSlot, p_bytes, peer_pbar + 8u * ps);
          bulk_copy_to_peer(peer_side + ps * kSideSlot, base + kOffSideOut + ps * kSideSlot, kSideSlot,
                            peer_pbar + 8u * ps);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------- QK issuer + rope-query loader
    // One thread; it blocks on its barriers (no polling), so the warps that
    // share its scheduler keep their issue slots.
    if (lane == 0) {
      tma_prefetch_desc(&tm_qr);
      const uint64_t dk = sdesc(base + kOffLat, 16, 1024);         // latent block 0, K-major (B of QK)
      const uint64_t dr = sdesc(base + kOffRope, 16, 512, kLayoutSw64);   // rope slot 0 (B of QK)
      const uint64_t dqr = sdesc(base + kOffQR, 16, 512, kLayoutSw64);    // rope query (A of QK)
      auto D = [](uint64_t d, uint32_t byte_off) -> uint64_t { return d + (byte_off >> 4); };
      uint32_t g = 0, nitem = 0;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
        if (!item_ok(p, nnz, b, s, e)) continue;
        const int nt = (e - s + T - 1) / T;
        // the rope query of this item replaces the previous one once its last QK is done
        if (nitem > 0 && !mbar_wait(bar(bQEmpty), (nitem - 1) & 1, wc)) break;
        // rows 0..H/2-1: this CTA's heads; rows 64..64+H/2-1: the peer's
        mbar_arrive_expect_tx(bar(bQFull), H * 64);
        tma_load_2d(base + kOffQR, &tm_qr, 32 * static_cast<int>(cta), b * H + static_cast<int>(cta) * Hh,
                    bar(bQFull));
        tma_load_2d(base + kOffQR + 64 * 64, &tm_qr, 32 * static_cast<int>(cta), b * H + static_cast<int>(peer) * Hh,
                    bar(bQFull));
        if (!mbar_wait(bar(bQFull), nitem & 1, wc)) break;     // + the latent half in TMEM
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t d_s = tmem + kTmS + (g & 1) * 64;
          const uint32_t blk = g % kLatBlocks, rs = g % kRopeSlots;
          if (g >= 2 && !mbar_wait(bar(bSFree + (g & 1)), ((g >> 1) - 1) & 1, wc)) { ok = false; break; }
          if (!mbar_wait(bar(bLatFull + blk), (g / kLatBlocks) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          MLA_TRACE_EVENT(2, g);
          const uint64_t bk = D(dk, blk * kLatBlock);
#pragma unroll
          for (int k = 0; k < 16; ++k)            // 256 latent dims = 16 K-steps; A (query) from TMEM
            umma_ts(d_s, tmem + kTmQ + 8 * k, D(bk, (k >> 2) * kAtom + (k & 3) * 32), kIdescQK, k != 0 ? 1u : 0u);
          if (!mbar_wait(bar(bRopeFull + rs), (g / kRopeSlots) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint64_t br = D(dr, rs * kRopeAtom);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)          // this CTA's half of the rope dims: 2 K-steps of 16
            umma_ss(d_s, D(dqr, kk * 32), D(br, kk * 32), kIdescQK, 1u);
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
  } else if (warp == kPvWarp) {
    // ------------------------------------------------- PV issuer + P copier
    if (lane == 0) {
      const uint64_t dv = sdesc(base + kOffLat, kAtom, 1024);      // latent block 0, MN-major (B of PV)
      const uint64_t dp = sdesc(base + kOffP, 16, 1024);           // P slot 0 (A of PV)
      auto D = [](uint64_t d, uint32_t byte_off) -> uint64_t { return d + (byte_off >> 4); };
      const uint16_t peer_mask = static_cast<uint16_t>(1u << peer);
      uint32_t g = 0, nitem = 0;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2];
        if (!item_ok(p, nnz, b, s, e)) continue;
        const int nt = (e - s + T - 1) / T;
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t ps = g % kPSlots, blk = g % kLatBlocks, use = g / kPSlots;
          if (!mbar_wait(bar(bPFull + ps), use & 1, wc)) { ok = false; break; }       // own P rows (and O rescaled)
          MLA_TRACE_EVENT(4, g);
          if (!mbar_wait(bar(bPeerOK + ps), use & 1, wc)) { ok = false; break; }      // the peer's P rows, applied
          if (j == 0 && nitem > 0 && !mbar_wait(bar(bOEmpty), (nitem - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bv = D(dv, blk * kLatBlock);
          const uint64_t ap = D(dp, ps * kPSlot);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)          // 64 tokens = 4 K-steps of 16
            umma_ss(tmem + kTmO, D(ap, ks * 32), D(bv, ks * 2048), kIdescPV, (j == 0 && ks == 0) ? 0u : 1u);
          umma_commit(bar(bLatEmpty + blk));
          umma_commit(bar(bPSlotMine + ps));
          umma_commit_mc(bar(bPSlotPeer + ps), peer_mask);     // in the peer: "the peer's PV of slot ps is done"
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
    // ------------------------------------------------- row warps and takers
    // Row warp w < 16: lane quadrant w & 3, token group / column quarter w >> 2.
    // Taker warps 18 and 19: lane quadrants 2 and 3, all 256 columns.
    const bool taker = warp >= kTakeWarp0;
    const int q = warp & 3, kg = taker ? 0 : warp >> 2;
    const bool own = q < 2;
    const int r = 32 * q + lane;                 // TMEM lane, P row, O row
    const int rl = own ? r : r - 64;             // row within the own or the peer half
    const int h = row_head(r, cta, Hh);          // head of this row, -1 for padding
    const bool row_ok = h >= 0;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    float* red_max = reinterpret_cast<float*>(smem + kOffRed);           // [2][4][64]
    float* red_l = red_max + 2 * 4 * 64;                                 // [4][64]
    const float* side = reinterpret_cast<const float*>(smem + kOffSide);
    auto wait = [&](uint32_t bb, uint32_t par, bool cluster_scope) {
      if (aborted) return;
      bool ok = true;
      if (lane == 0) ok = cluster_scope ? mbar_wait<true>(bb, par, wc) : mbar_wait(bb, par, wc);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) aborted = true;
    };
    // PV(g) has completed (this CTA)
    auto wait_pv = [&](uint32_t g) { wait(bar(bPSlotMine + (g % kPSlots)), (g / kPSlots) & 1, false); };
    // O row r, columns [c0, c0 + 16 n), times alpha (after PV(g-1))
    auto rescale_o = [&](float alpha, int c0, int n) {
      if (aborted) return;
#pragma unroll 1
      for (int c = 0; c < n; ++c) {
        uint32_t o[16];
        const uint32_t ta = tmem + lane_off + kTmO + c0 + 16 * c;
        tmem_ld16(ta, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st16(ta, o);
      }
      tmem_wait_st();
    };
    // the usable items, walked by every role in the same order
    auto next_ok = [&](int i) {
      for (; i < it1; ++i) {
        const int b = items[4 * i], s = items[4 * i + 1], e = items[4 * i + 2];
        if (item_ok(p, nnz, b, s, e)) return i;
      }
      return it1;
    };

    if (taker) {
      // ---------------------------------------------------------- takers
      // tile g: once the peer's P rows have landed, apply its rescale factors
      // to these 32 rows of O (all 256 columns); PV(g) waits for this
      // (an item's last tile also brings the peer's row sums: they are kept
      // here, per item parity, for the pushers' write-out after its last PV)
      float* l_peer = reinterpret_cast<float*>(smem + kOffLPeer);
      uint32_t g = 0, nitem = 0;
      for (int it = next_ok(it0); it < it1; it = next_ok(it + 1), ++nitem) {
        const int s = items[4 * it + 1], e = items[4 * it + 2];
        const int nt = (e - s + T - 1) / T;
        for (int j = 0; j < nt; ++j, ++g) {
          const uint32_t ps = g % kPSlots;
          // arm the slot for the peer's P rows and side slot of tile g: by the
          // taker that also waits on it, so never before tile g - 2's phase
          // has completed (the bytes may land either side of the arm)
          if (warp == kTakeWarp0 && lane == 0 && !aborted)
            mbar_arrive_expect_tx(bar(bPeerP + ps), static_cast<uint32_t>(Hh) * 128u + kSideSlot);
          wait(bar(bPeerP + ps), (g / kPSlots) & 1, true);
          if (lane == 0 && warp == kTakeWarp0) MLA_TRACE_EVENT(13, g);
          if (j == nt - 1 && row_ok && !aborted)
            l_peer[(nitem & 1) * 64 + rl] = side[ps * (kSideSlot / 4) + 64 + rl];
          const float alpha = (!aborted && row_ok) ? side[ps * (kSideSlot / 4) + rl] : 1.f;
          if (__any_sync(0xffffffffu, alpha != 1.f)) {   // never on an item's first tile
            wait_pv(g - 1);
            tc_fence_after();
            rescale_o(alpha, 0, 16);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0 && !aborted) mbar_arrive(bar(bPeerOK + ps));
        }
      }
    } else {
      // -------------------------------------------------------- row warps
      // -- this warp's 16 S columns of tile g (raw fp32 partial), then free the S buffer
      auto read_s = [&](uint32_t g, uint32_t (&v)[16]) {
        const uint32_t sb = g & 1;
        wait(bar(bSFull + sb), (g >> 1) & 1, false);
        if (!aborted) {
          tc_fence_after();
          tmem_ld16(tmem + lane_off + kTmS + sb * 64 + kg * kGroup, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(bSFree + sb));
      };

      // -- the latent half of the query of request b for this warp's row and 64 dims, into TMEM
      auto load_q = [&](int b) {
        if (!aborted) {
          const uint4* src = reinterpret_cast<const uint4*>(
              p.q_nope + (static_cast<size_t>(b) * H + (row_ok ? h : 0)) * kLatent + 256 * cta + 64 * kg);
#pragma unroll
          for (int c = 0; c < 2; ++c) {          // 2 x 16 columns = 64 bf16
            uint32_t v16[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint4 v = row_ok ? __ldg(src + 4 * c + k) : make_uint4(0, 0, 0, 0);
              v16[4 * k] = v.x; v16[4 * k + 1] = v.y; v16[4 * k + 2] = v.z; v16[4 * k + 3] = v.w;
            }
            tmem_st16(tmem + lane_off + kTmQ + 32 * kg + 16 * c, v16);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(bQFull));
      };

      // -- after an item's last PV: O row r (this warp's 64 columns) / l to out or a partial state
      const float* l_peer = reinterpret_cast<const float*>(smem + kOffLPeer);
      auto write_o = [&](int b, int part, uint32_t nitem, float lsum, float lse_val) {
        wait(bar(bOFull), nitem & 1, false);
        tc_fence_after();
        // the peer's row sum of a peer row: stored by the takers before they
        // released the item's last PV, which bOFull follows
        if (!own) lsum = (!aborted && row_ok) ? l_peer[(nitem & 1) * 64 + rl] : 0.f;
        const bool part_ok = part < p.max_partials;   // a device-only plan naming a partial past the workspace
        if (!part_ok && threadIdx.x == 0) record_status(p.status, MLA_ERR_PLAN_MISMATCH);
        if (!aborted && part_ok) {
          const float inv = lsum > 0.f ? 1.f / lsum : 0.f;     // no valid score: out = 0
          float* dst_f = nullptr;
          __nv_bfloat16* dst_h = nullptr;
          const size_t col0 = 256 * static_cast<size_t>(cta) + 64 * kg;
          const size_t hh = row_ok ? static_cast<size_t>(h) : 0;
          if (part < 0) {
            const size_t o = (static_cast<size_t>(b) * H + hh) * kLatent + col0;
            if (p.out_bf16) dst_h = reinterpret_cast<__nv_bfloat16*>(p.out) + o;
            else dst_f = reinterpret_cast<float*>(p.out) + o;
          } else {
            dst_f = p.part_o + (static_cast<size_t>(part) * H + hh) * kLatent + col0;
          }
#pragma unroll 1
          for (int cb = 0; cb < 2; ++cb) {        // 32 columns per TMEM round trip, 32-byte stores
            uint32_t o[32];
            {
              uint32_t a[16], c[16];
              tmem_ld16(tmem + lane_off + kTmO + 64 * kg + 32 * cb, a);
              tmem_ld16(tmem + lane_off + kTmO + 64 * kg + 32 * cb + 16, c);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) { o[i] = a[i]; o[16 + i] = c[i]; }
            }
            if (row_ok) {
              if (dst_f) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  uint32_t v[8];
#pragma unroll
                  for (int k = 0; k < 8; ++k) v[k] = __float_as_uint(__uint_as_float(o[8 * i + k]) * inv);
                  st_global_v8(dst_f + 32 * cb + 8 * i, v);
                }
              } else {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                  uint32_t v[8];
#pragma unroll
                  for (int k = 0; k < 8; ++k)
                    v[k] = pack_bf16x2(__uint_as_float(o[16 * i + 2 * k]) * inv,
                                       __uint_as_float(o[16 * i + 2 * k + 1]) * inv);
                  st_global_v8(dst_h + 32 * cb + 16 * i, v);
                }
              }
            }
          }
          if (own && kg == 0 && row_ok) {          // the owner of the head writes its lse
            if (part < 0) { if (p.lse) p.lse[static_cast<size_t>(b) * H + h] = lse_val; }
            else p.part_lse[static_cast<size_t>(part) * H + h] = lse_val;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(bar(bOEmpty));
      };

      // an item's output is written after the next item's first tile, so that
      // the epilogue overlaps that tile's exchange instead of delaying it
      struct Pending { int b, part; uint32_t nitem; float lsum, lse; };
      Pending pend{-1, 0, 0, 0.f, 0.f};
      auto flush = [&]() {
        if (pend.b < 0) return;
        write_o(pend.b, pend.part, pend.nitem, pend.lsum, pend.lse);
        pend.b = -1;
      };

      int it = next_ok(it0);
      if (it < it1) load_q(items[4 * it]);      // the first item's query
      uint32_t g = 0, nitem = 0;

      if (own) {
        // ---------------------------------------------- softmax (own rows)
        float* side_out = reinterpret_cast<float*>(smem + kOffSideOut);   // [kPSlots][alpha 64 | l 64]
        float m_ref = 0.f, l_sum = 0.f, lsum = 0.f;
        for (; it < it1; it = next_ok(it + 1)) {
          const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2], part = items[4 * it + 3];
          const int n = e - s, nt = (n + T - 1) / T;
          // multi-query: head h is query h / (H / q_len) of its request, which
          // sees the first L - q_len + 1 + i rows of the request's context
          int n_row = n;
          if (p.q_len > 1 && row_ok) {
            const int lo = __ldg(p.kv_indptr + b), hi = __ldg(p.kv_indptr + b + 1);
            const int i = h / (H / p.q_len);
            n_row = max(0, min(n, (hi - lo) - p.q_len + 1 + i - (s - lo)));
          }
          for (int j = 0; j < nt; ++j, ++g) {
            const uint32_t xs = g % kXSlots, ps = g % kPSlots;
            // arm the receive slot for the peer's partials of tile g: done here,
            // by a warp that also waits on it, so the arm for tile g + kXSlots
            // cannot come before this tile's phase has completed
            if (warp == 0 && lane == 0 && !aborted)
              mbar_arrive_expect_tx(bar(bXFull + xs), static_cast<uint32_t>(Hh) * T * 4u);
            uint32_t sv[16];
            read_s(g, sv);
            if (threadIdx.x == 0) MLA_TRACE_EVENT(10, g);
            wait(bar(bXFull + xs), (g / kXSlots) & 1, true);
            if (threadIdx.x == 0) MLA_TRACE_EVENT(9, g);
            // s = (own + peer) * sm_scale * log2(e): the full score as an fp32 sum of the two halves
            {
              const uint8_t* xrow = smem + kOffX + xs * kXSlot + rl * 256;
              const float2 sl2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint32_t c = static_cast<uint32_t>(4 * kg + i);
                uint4 pv = make_uint4(0, 0, 0, 0);
                if (!aborted) pv = *reinterpret_cast<const uint4*>(xrow + ((c ^ static_cast<uint32_t>(rl & 15)) << 4));
                const float2 a = f2_mul(f2_add(f2_pack(__uint_as_float(sv[4 * i]), __uint_as_float(sv[4 * i + 1])),
                                               f2_pack(__uint_as_float(pv.x), __uint_as_float(pv.y))), sl2);
                const float2 c2 = f2_mul(f2_add(f2_pack(__uint_as_float(sv[4 * i + 2]), __uint_as_float(sv[4 * i + 3])),
                                                f2_pack(__uint_as_float(pv.z), __uint_as_float(pv.w))), sl2);
                sv[4 * i] = __float_as_uint(a.x);
                sv[4 * i + 1] = __float_as_uint(a.y);
                sv[4 * i + 2] = __float_as_uint(c2.x);
                sv[4 * i + 3] = __float_as_uint(c2.y);
              }
            }
            if (threadIdx.x == 0) MLA_TRACE_EVENT(1, g);
            const int nvalid = n_row - j * T - kg * kGroup;
            if (nvalid < kGroup) {
#pragma unroll
              for (int t = 0; t < kGroup; ++t)
                if (t >= nvalid) sv[t] = __float_as_uint(-INFINITY);
            }
            const float mh =
                fmaxf(max3(max3(__uint_as_float(sv[0]), __uint_as_float(sv[1]), __uint_as_float(sv[2])),
                           max3(__uint_as_float(sv[3]), __uint_as_float(sv[4]), __uint_as_float(sv[5])),
                           max3(__uint_as_float(sv[6]), __uint_as_float(sv[7]), __uint_as_float(sv[8]))),
                      max3(max3(__uint_as_float(sv[9]), __uint_as_float(sv[10]), __uint_as_float(sv[11])),
                           max3(__uint_as_float(sv[12]), __uint_as_float(sv[13]), __uint_as_float(sv[14])),
                           __uint_as_float(sv[15])));
            // row maximum over the tile: the four warps of the quadrant
            float* rm = red_max + (g & 1) * 256;
            rm[kg * 64 + r] = mh;
            named_bar_sync(1 + q, 128);
            const float mt = fmaxf(fmaxf(rm[r], rm[64 + r]), fmaxf(rm[128 + r], rm[192 + r]));
            float alpha = 1.f;
            if (j == 0 || m_ref == -INFINITY) {
              // an item's first tile sets the reference; so does the first tile
              // with a valid score when a causal query row had none before (O and
              // the row sum are still zero then)
              m_ref = mt;
              if (j == 0) l_sum = 0.f;
            } else {
              const bool need = mt > m_ref + 64.f;
              if (__any_sync(0xffffffffu, need)) {
                wait_pv(g - 1);                      // PV(g-1) must have landed before O is rescaled
                tc_fence_after();
                if (need) {
                  alpha = ex2_approx(m_ref - mt);
                  m_ref = mt;
                  l_sum *= alpha;
                }
                rescale_o(alpha, 64 * kg, 4);
                tc_fence_before();
              }
            }
            if (threadIdx.x == 0) MLA_TRACE_EVENT(11, g);
            // P = 2^(s - m_ref) as bf16 into P slot ps (K-major, 128-byte swizzle),
            // once both CTAs' PVs of tile g - kPSlots have read it (this CTA's
            // own rows, and the peer's copy of them)
            if (g >= static_cast<uint32_t>(kPSlots)) {
              wait_pv(g - kPSlots);
              wait(bar(bPSlotPeer + ps), ((g / kPSlots) - 1) & 1, true);
            }
            if (threadIdx.x == 0) MLA_TRACE_EVENT(12, g);
            const float m_eff = m_ref == -INFINITY ? 0.f : m_ref;   // a row with no valid score yet: P = 0
            const float2 nm2 = f2_pack(-m_eff, -m_eff);
            float2 l4[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
            uint8_t* prow = smem + kOffP + ps * kPSlot + r * 128;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t pk[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 d =
                    f2_add(f2_pack(__uint_as_float(sv[8 * c + 2 * i]), __uint_as_float(sv[8 * c + 2 * i + 1])), nm2);
                const float a0 = ex2_approx(d.x), a1 = ex2_approx(d.y);
                l4[i & 1] = f2_add(l4[i & 1], f2_pack(a0, a1));
                pk[i] = pack_bf16x2(a0, a1);
              }
              const uint32_t ch = static_cast<uint32_t>(2 * kg + c);
              if (!aborted)
                *reinterpret_cast<uint4*>(prow + ((ch ^ static_cast<uint32_t>(r & 7)) << 4)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            const float2 l2 = f2_add(l4[0], l4[1]);
            l_sum += l2.x + l2.y;
            // this row's rescale factor and, after an item's last tile, its row
            // sum (the four warps' parts added in a fixed order), for the
            // peer's half of O: they travel with the P rows
            if (kg == 0 && !aborted) side_out[ps * (kSideSlot / 4) + rl] = alpha;
            if (j == nt - 1) {
              red_l[kg * 64 + r] = l_sum;
              named_bar_sync(1 + q, 128);
              lsum = (red_l[r] + red_l[64 + r]) + (red_l[128 + r] + red_l[192 + r]);
              if (kg == 0 && !aborted) side_out[ps * (kSideSlot / 4) + 64 + rl] = lsum;
            }
            if (threadIdx.x == 0) MLA_TRACE_EVENT(14, g);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && !aborted) mbar_arrive(bar(bPFull + ps));
            if (threadIdx.x == 0) MLA_TRACE_EVENT(7, g);
            if (j == 0) flush();                   // the previous item's output
          }
          // (red_l is rewritten at the next item's last tile, after at least one
          // more tile-maximum barrier, so every warp has read it by then)
          const float lse_val = lsum > 0.f ? (m_ref + __log2f(lsum)) * 0.69314718055994531f : -INFINITY;
          // the next item's query, as soon as this item's last QK is done
          const int nx = next_ok(it + 1);
          if (nx < it1) {
            wait(bar(bQEmpty), nitem & 1, false);
            tc_fence_after();
            load_q(items[4 * nx]);
          }
          pend = Pending{b, part, nitem, lsum, lse_val};
          ++nitem;
        }
        flush();
      } else {
        // ----------------------------------------- pushers (the peer's rows)
        const uint32_t xrow_peer = mapa_shared(base + kOffX + rl * 256, peer);
        const uint32_t xfull_peer = mapa_shared(bar(bXFull), peer);
        for (; it < it1; it = next_ok(it + 1)) {
          const int b = items[4 * it], s = items[4 * it + 1], e = items[4 * it + 2], part = items[4 * it + 3];
          const int nt = (e - s + T - 1) / T;
          for (int j = 0; j < nt; ++j, ++g) {
            // tile g: this CTA's partial of the peer's row into the peer's receive slot
            const uint32_t xs = g % kXSlots;
            uint32_t v[16];
            read_s(g, v);
            if (threadIdx.x == 64) MLA_TRACE_EVENT(6, g);
            if (g >= static_cast<uint32_t>(kXSlots)) wait(bar(bXFree + xs), ((g / kXSlots) - 1) & 1, true);
            if (row_ok && !aborted) {
              const uint32_t dst = xrow_peer + xs * kXSlot, fb = xfull_peer + 8u * xs;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint32_t c = static_cast<uint32_t>(4 * kg + i);
                st_async_v4(dst + ((c ^ static_cast<uint32_t>(rl & 15)) << 4), v[4 * i], v[4 * i + 1], v[4 * i + 2],
                            v[4 * i + 3], fb);
              }
            }
            if (threadIdx.x == 64) MLA_TRACE_EVENT(8, g);
            if (j == 0) flush();                   // the previous item's output
          }
          const int nx = next_ok(it + 1);
          if (nx < it1) {
            wait(bar(bQEmpty), nitem & 1, false);
            tc_fence_after();
            load_q(items[4 * nx]);
          }
          pend = Pending{b, part, nitem, 0.f, 0.f};
          ++nitem;
        }
        flush();
      }
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
  if (warp == kPvWarp) tmem_dealloc(tmem, 512);
}

}  // namespace pair

int launch_pair(int heads, const CUtensorMap& tm_kv, const CUtensorMap& tm_kv_rope, const CUtensorMap& tm_qr,
                const DecodeParams& p, int workers, cudaStream_t stream) {
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
  if (cudaLaunchKernelEx(&cfg, pair::pair_kernel, tm_kv, tm_kv_rope, tm_qr, p) != cudaSuccess) return MLA_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace mla
