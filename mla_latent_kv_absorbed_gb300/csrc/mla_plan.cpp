// Host-side split-KV plan: choose per-request chunking and place the chunks on
// the SMs.  ("Attention backends", paragraph "Paged, ragged batches": the CSR
// arrays are rebuilt on the CPU for each batch, and plan() picks the split-KV
// chunking per request and balances long and short contexts across SMs.  The
// page states the goal, not a rule; the rule below is this library's.)
//
//   * variant by head count: H in {16, 32} -> one CTA per worker; H in
//     48..128 (step 16) -> a 2-CTA cluster per worker; 64-token tiles for both;
//   * W workers = SMs / CTAs-per-worker;
//   * candidate chunk sizes c_k = max(1, ceil(ceil(total_tiles / W) / k)),
//     k = 1..8, duplicates dropped;
//   * a request of t tiles becomes ceil(t / c) chunks; chunk cost = tiles + 1;
//   * longest-processing-time placement: chunks sorted by (cost desc, request,
//     chunk index), each to the least-loaded worker (ties: lowest index);
//   * objective = makespan + 4 if any request was cut; smallest wins, ties to
//     the earlier (larger) candidate.
// The plan is deterministic: equal inputs give identical words.
#include <algorithm>
#include <cstdint>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "mla_plan.h"

namespace mla {

namespace {

struct Chunk {
  int b;
  int k;
  int tiles;
};

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

void make_chunks(const std::vector<long long>& tiles, long long c, std::vector<Chunk>& out) {
  out.clear();
  for (size_t b = 0; b < tiles.size(); ++b) {
    const long long t = tiles[b];
    if (t <= 0) continue;
    const long long n = ceil_div(t, c);
    for (long long k = 0; k < n; ++k)
      out.push_back({static_cast<int>(b), static_cast<int>(k), static_cast<int>(std::min(c, t - k * c))});
  }
}

// LPT placement; returns the makespan and fills per-worker lists.
long long place(std::vector<Chunk> chunks, int W, std::vector<std::vector<Chunk>>& lists) {
  std::sort(chunks.begin(), chunks.end(), [](const Chunk& x, const Chunk& y) {
    if (x.tiles != y.tiles) return x.tiles > y.tiles;   // cost = tiles + const
    if (x.b != y.b) return x.b < y.b;
    return x.k < y.k;
  });
  using Slot = std::pair<long long, int>;   // (load, worker)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int w = 0; w < W; ++w) heap.push({0, w});
  lists.assign(W, {});
  for (const Chunk& ch : chunks) {
    Slot s = heap.top();
    heap.pop();
    lists[s.second].push_back(ch);
    s.first += ch.tiles + kItemOverheadTiles;
    heap.push(s);
  }
  long long makespan = 0;
  while (!heap.empty()) {
    makespan = std::max(makespan, heap.top().first);
    heap.pop();
  }
  return makespan;
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

  std::vector<long long> tiles(B);
  long long total = 0;
  for (int b = 0; b < B; ++b) {
    const long long L = static_cast<long long>(indptr[b + 1]) - indptr[b];
    tiles[b] = ceil_div(L, T);
    total += tiles[b];
  }

  long long c = 1;
  std::vector<std::vector<Chunk>> lists(W);
  if (total > 0) {
    const long long base = ceil_div(total, W);
    long long best_obj = -1;
    std::vector<long long> seen;
    std::vector<Chunk> chunks;
    std::vector<std::vector<Chunk>> cand;
    for (int k = 1; k <= kNumCandidates; ++k) {
      const long long cc = std::max<long long>(1, ceil_div(base, k));
      if (std::find(seen.begin(), seen.end(), cc) != seen.end()) continue;
      seen.push_back(cc);
      make_chunks(tiles, cc, chunks);
      const long long makespan = place(chunks, W, cand);
      bool cut = false;
      for (long long t : tiles) cut = cut || t > cc;
      const long long obj = makespan + (cut ? kMergeCostTiles : 0);
      if (best_obj < 0 || obj < best_obj) {
        best_obj = obj;
        c = cc;
        lists.swap(cand);
      }
    }
  }

  std::vector<long long> nchunks(B), pstart(B);
  long long P = 0;
  for (int b = 0; b < B; ++b) {
    nchunks[b] = tiles[b] > 0 ? ceil_div(tiles[b], c) : 0;
    pstart[b] = P;
    if (nchunks[b] > 1) P += nchunks[b];
  }

  std::vector<int32_t> wptr(1, 0), items;
  for (int w = 0; w < W; ++w) {
    for (const Chunk& ch : lists[w]) {
      const long long begin = static_cast<long long>(indptr[ch.b]) + static_cast<long long>(ch.k) * c * T;
      const long long end = std::min<long long>(indptr[ch.b + 1], begin + c * T);
      const long long part = nchunks[ch.b] > 1 ? pstart[ch.b] + ch.k : -1;
      items.push_back(ch.b);
      items.push_back(static_cast<int32_t>(begin));
      items.push_back(static_cast<int32_t>(end));
      items.push_back(static_cast<int32_t>(part));
    }
    wptr.push_back(static_cast<int32_t>(items.size() / 4));
  }
  std::vector<int32_t> merge;
  for (int b = 0; b < B; ++b) {
    if (nchunks[b] != 1) {
      merge.push_back(b);
      merge.push_back(static_cast<int32_t>(pstart[b]));
      merge.push_back(static_cast<int32_t>(pstart[b] + (nchunks[b] > 1 ? nchunks[b] : 0)));
    }
  }
  const long long n_items = static_cast<long long>(items.size() / 4);
  const long long n_merge = static_cast<long long>(merge.size() / 3);
  const long long total_words = kHeaderWords + (W + 1) + 4 * n_items + 3 * n_merge;
  if (total_words > (1ll << 31) - 1 || P > (1ll << 31) - 1) return MLA_ERR_INVALID_ARG;

  words.assign(kHeaderWords, 0);
  words[kHMagic] = kPlanMagic;
  words[kHVersion] = kPlanVersion;
  words[kHBatch] = B;
  words[kHHeads] = H;
  words[kHVariant] = variant;
  words[kHTile] = T;
  words[kHWorkers] = W;
  words[kHChunkTiles] = static_cast<int32_t>(c);
  words[kHItems] = static_cast<int32_t>(n_items);
  words[kHPartials] = static_cast<int32_t>(P);
  words[kHMerges] = static_cast<int32_t>(n_merge);
  words[kHHeadGroups] = 1;
  words[kHCtasPerWorker] = cpw;
  words[kHTotalWords] = static_cast<int32_t>(total_words);
  words[kHNumSms] = num_sms;
  words[kHReserved] = 0;
  words.insert(words.end(), wptr.begin(), wptr.end());
  words.insert(words.end(), items.begin(), items.end());
  words.insert(words.end(), merge.begin(), merge.end());

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

}  // namespace mla
