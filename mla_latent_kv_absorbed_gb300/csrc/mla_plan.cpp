// Host-side split-KV plan: choose per-request chunking and place the chunks on
// the SMs.  ("Attention backends", paragraph "Paged, ragged batches": the CSR
// arrays are rebuilt on the CPU for each batch, and plan() picks the split-KV
// chunking per request and balances long and short contexts across SMs.  The
// page states the goal, not a rule; the rule below is this library's.)
//
//   * variant by head count: H in {16, 32} -> one CTA per worker; H in
//     48..128 (step 16) -> a 2-CTA cluster per worker; 64-token tiles for both;
//   * W workers = SMs / CTAs-per-worker; loads are counted in tokens, an item
//     of n tokens costs its tiles, roundup(n, 64), plus the variant's item
//     overhead (its epilogue and the refill behind it: 32 tokens for one-CTA
//     workers, 256 for two-CTA workers): a worker's time follows its tiles,
//     ragged or not, and its items;
//   * wrap-around fill: requests, in order, are poured into workers 0, 1, ...
//     each up to a load budget cap, so a request is cut only where a worker
//     is full (at most W - 1 cuts, hence few partial states to merge), at a
//     tile boundary of the request (only its last piece has a ragged tile);
//   * no cut piece is shorter than kMinPieceTokens and no worker's load
//     exceeds cap: where the tail after the whole tiles that fit would be
//     shorter, the cut moves one tile earlier (the tail piece then holds a
//     whole tile besides its ragged one; a worker one tile over cap would be
//     the step's slowest); with less space than that the worker is closed;
//   * cap starts at ceil((total + (nonempty + W - 1) * overhead) / W) tokens,
//     total counting every request in whole tiles, and grows by
//     kCapStepTokens until the fill fits on W workers.
// The plan is deterministic: equal inputs give identical words.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "mla_plan.h"

namespace mla {

namespace {

struct Piece {
  int w;             // worker
  int b;
  long long k0;      // first token of the piece inside its request
  long long n;       // tokens
};

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
constexpr long long kTileTokens = 64;
inline long long round_up_tile(long long n) { return ceil_div(n, kTileTokens) * kTileTokens; }

// Wrap-around fill with load budget cap (tokens); false when W workers do not
// suffice.  Pieces come out in worker order (the fill only moves forward), so
// one flat list holds them all: no allocation per attempt once it has grown.
bool fill(const std::vector<long long>& len, int W, long long cap, long long ov, std::vector<Piece>& pieces) {
  pieces.clear();
  int w = 0;
  long long used = 0;
  for (size_t b = 0; b < len.size(); ++b) {
    long long k0 = 0;
    const long long L = len[b];
    while (k0 < L) {
      if (w == W) return false;
      const long long rem = L - k0;
      const long long space = cap - used - ov;
      const long long fit = space / kTileTokens * kTileTokens;   // whole tiles that fit
      long long take;
      if (round_up_tile(rem) <= space) {
        take = rem;
      } else if (fit >= kMinPieceTokens && rem - fit >= kMinPieceTokens) {
        take = fit;
      } else if (fit - kTileTokens >= kMinPieceTokens) {
        take = fit - kTileTokens;                                  // the tail keeps a whole tile
      } else {
        ++w;
        used = 0;
        continue;
      }
      pieces.push_back({w, static_cast<int>(b), k0, take});
      used += round_up_tile(take) + ov;
      k0 += take;
    }
  }
  return true;
}

}  // namespace

int variant_for_heads(int H, int* tile, int* ctas_per_worker) {
  if (H == 16 || H == 32) {
    *tile = 64;
    *ctas_per_worker = 1;
    return kVariantSwab;
  }
  if (H >= 48 && H <= 128 && H % 16 == 0) {
    *tile = 64;
    *ctas_per_worker = 2;
    return kVariantPair;
  }
  return 0;
}

int build_plan(const int32_t* indptr, int B, int H, int num_sms, std::vector<int32_t>& words,
               size_t* workspace_bytes) {
  int T = 0, cpw = 0;
  const int variant = variant_for_heads(H, &T, &cpw);
  if (!variant) return MLA_ERR_UNSUPPORTED;
  const int W = num_sms / cpw;
  if (W < 1) return MLA_ERR_INVALID_ARG;

  std::vector<long long> len(B);
  long long total = 0, nonempty = 0;   // total in whole tiles
  for (int b = 0; b < B; ++b) {
    len[b] = static_cast<long long>(indptr[b + 1]) - indptr[b];
    total += round_up_tile(len[b]);
    nonempty += len[b] > 0 ? 1 : 0;
  }
  long long cap = 0;
  std::vector<Piece> pieces;
  pieces.reserve(static_cast<size_t>(B) + W);
  if (total > 0) {
    const long long ov = item_overhead_tokens(variant);
    cap = ceil_div(total + (nonempty + W - 1) * ov, W);
    while (!fill(len, W, cap, ov, pieces)) cap += kCapStepTokens;
  }

  // per request: pieces, first partial index, pieces numbered so far (one allocation)
  std::vector<long long> acc(3 * static_cast<size_t>(B), 0);
  long long* npieces = acc.data();
  long long* pstart = npieces + B;
  long long* seen = pstart + B;
  for (const Piece& pc : pieces) ++npieces[pc.b];
  long long P = 0, n_merge = 0;
  for (int b = 0; b < B; ++b) {
    pstart[b] = P;
    if (npieces[b] > 1) P += npieces[b];
    if (npieces[b] != 1) ++n_merge;
  }
  const long long n_items = static_cast<long long>(pieces.size());
  const long long total_words = kHeaderWords + (W + 1) + 4 * n_items + 3 * n_merge;
  if (total_words > (1ll << 31) - 1 || P > (1ll << 31) - 1) return MLA_ERR_INVALID_ARG;

  // the words are written in place: header, worker_indptr, items, merge entries
  words.assign(static_cast<size_t>(total_words), 0);
  int32_t* hw = words.data();
  hw[kHMagic] = kPlanMagic;
  hw[kHVersion] = kPlanVersion;
  hw[kHBatch] = B;
  hw[kHHeads] = H;
  hw[kHVariant] = variant;
  hw[kHTile] = T;
  hw[kHWorkers] = W;
  hw[kHCap] = static_cast<int32_t>(cap);
  hw[kHItems] = static_cast<int32_t>(n_items);
  hw[kHPartials] = static_cast<int32_t>(P);
  hw[kHMerges] = static_cast<int32_t>(n_merge);
  hw[kHHeadGroups] = 1;
  hw[kHCtasPerWorker] = cpw;
  hw[kHTotalWords] = static_cast<int32_t>(total_words);
  hw[kHNumSms] = num_sms;
  hw[kHReserved] = 0;
  int32_t* wptr = hw + kHeaderWords;
  int32_t* items = wptr + W + 1;
  int32_t* merge = items + 4 * n_items;
  wptr[0] = 0;
  size_t pi = 0;
  for (int w = 0; w < W; ++w) {
    for (; pi < pieces.size() && pieces[pi].w == w; ++pi) {
      const Piece& pc = pieces[pi];
      const long long begin = static_cast<long long>(indptr[pc.b]) + pc.k0;
      const long long end = begin + pc.n;
      const long long part = npieces[pc.b] > 1 ? pstart[pc.b] + seen[pc.b] : -1;
      ++seen[pc.b];
      int32_t* itw = items + 4 * pi;
      itw[0] = pc.b;
      itw[1] = static_cast<int32_t>(begin);
      itw[2] = static_cast<int32_t>(end);
      itw[3] = static_cast<int32_t>(part);
    }
    wptr[w + 1] = static_cast<int32_t>(pi);
  }
  for (int b = 0; b < B; ++b) {
    if (npieces[b] != 1) {
      merge[0] = b;
      merge[1] = static_cast<int32_t>(pstart[b]);
      merge[2] = static_cast<int32_t>(pstart[b] + (npieces[b] > 1 ? npieces[b] : 0));
      merge += 3;
    }
  }

  size_t ws = kWsHeaderBytes + static_cast<size_t>(P) * H * kLatent * 4 + static_cast<size_t>(P) * H * 4;
  ws = (ws + 255) / 256 * 256;
  *workspace_bytes = ws;
  return MLA_OK;
}

// Offsets of the partial arrays inside the workspace.
size_t ws_part_o_offset() { return kWsHeaderBytes; }
size_t ws_part_lse_offset(const int32_t* header) {
  return kWsHeaderBytes + static_cast<size_t>(header[kHPartials]) * header[kHHeads] * kLatent * 4;
}
size_t ws_needed_bytes(const int32_t* header) {
  return ws_part_lse_offset(header) + static_cast<size_t>(header[kHPartials]) * header[kHHeads] * 4;
}

}  // namespace mla
