"""Plain restatement of the split-KV decode plan (host integer logic).

TEST INFRASTRUCTURE ONLY.  Only ``tests/`` and ``__graft_entry__.smoke()`` may
import this module.  It shares no code with the library's C++ plan; the tests
compare the two word for word.

The pages fix only the plan's job: "Attention backends", paragraph "Paged,
ragged batches" -- the CSR arrays are rebuilt on the CPU for each batch and
plan() chooses the split-KV chunking per request and balances long and short
contexts across SMs.  They give no rule, so this is the one the library uses:

  * kernel variant by head count: H in {16, 32} -> "swab" (one CTA per SM);
    H in {48, 64, ..., 128} -> "pair" (a two-CTA cluster per worker); both
    work in 64-token tiles;
  * W workers = SMs (swab) or SMs // 2 (pair);
  * tiles_b = ceil(L_b / T); total = sum tiles_b; base = ceil(total / W);
  * candidate chunk sizes (in tiles) c_k = max(1, ceil(base / k)), k = 1..8,
    duplicates dropped, in that order;
  * for a candidate c, request b with tiles_b > 0 is cut into
    ceil(tiles_b / c) chunks of c tiles (the last one shorter); each chunk is a
    work item of cost tiles + ITEM_OVERHEAD;
  * items are placed longest-processing-time first: sorted by
    (-cost, b, chunk), each goes to the worker with the smallest load, ties to
    the lowest worker index;
  * objective = makespan + (MERGE_COST if any request is cut, else 0);
    the smallest objective wins, ties to the earlier candidate;
  * partial slots are numbered over the cut requests in (b, chunk) order; an
    uncut request's item writes out/lse directly (partial = -1);
  * the merge list holds every request that is cut or empty, in b order, with
    its partial range (empty requests get an empty range).

Plan words (int32): a 16-word header, worker_indptr[W+1], 4 words per item
(b, kv_begin, kv_end, partial) grouped by worker in placement order, then 3
words per merge entry (b, p_begin, p_end).
"""
from __future__ import annotations

import heapq

PLAN_MAGIC = 0x4D4C4131
PLAN_VERSION = 1
HEADER_WORDS = 16
ITEM_OVERHEAD = 1
MERGE_COST = 4
NUM_CANDIDATES = 8
WS_HEADER_BYTES = 256
D_LATENT = 512

VARIANT_SWAB = 1
VARIANT_PAIR = 2


def variant_for_heads(H: int):
    """(variant, tile_tokens, ctas_per_worker) or None when H is unsupported."""
    if H in (16, 32):
        return VARIANT_SWAB, 64, 1
    if 48 <= H <= 128 and H % 16 == 0:
        return VARIANT_PAIR, 64, 2
    return None


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def _chunks(tiles, c):
    items = []
    for b, t in enumerate(tiles):
        n = _ceil_div(t, c) if t > 0 else 0
        for k in range(n):
            items.append((b, k, min(c, t - k * c)))
    return items


def _place(items, W):
    """LPT placement. Returns (makespan, per-worker item lists)."""
    order = sorted(items, key=lambda it: (-(it[2] + ITEM_OVERHEAD), it[0], it[1]))
    heap = [(0, w) for w in range(W)]
    lists = [[] for _ in range(W)]
    for it in order:
        load, w = heapq.heappop(heap)
        lists[w].append(it)
        heapq.heappush(heap, (load + it[2] + ITEM_OVERHEAD, w))
    makespan = max(load for load, _ in heap) if heap else 0
    return makespan, lists


def build_plan(kv_indptr, H: int, num_sms: int):
    """Returns (plan words as a list of ints, workspace bytes)."""
    v = variant_for_heads(H)
    if v is None:
        raise ValueError("unsupported head count")
    variant, T, cpw = v
    B = len(kv_indptr) - 1
    lengths = [int(kv_indptr[b + 1]) - int(kv_indptr[b]) for b in range(B)]
    W = num_sms // cpw
    if W < 1:
        raise ValueError("too few SMs")
    tiles = [_ceil_div(L, T) for L in lengths]
    total = sum(tiles)

    best = None
    if total > 0:
        base = _ceil_div(total, W)
        seen = []
        for k in range(1, NUM_CANDIDATES + 1):
            c = max(1, _ceil_div(base, k))
            if c in seen:
                continue
            seen.append(c)
            items = _chunks(tiles, c)
            makespan, lists = _place(items, W)
            cut = any(t > c for t in tiles)
            obj = makespan + (MERGE_COST if cut else 0)
            if best is None or obj < best[0]:
                best = (obj, c, lists)
        _, c, lists = best
    else:
        c, lists = 1, [[] for _ in range(W)]

    nchunks = [(_ceil_div(t, c) if t > 0 else 0) for t in tiles]
    pstart = []
    P = 0
    for b in range(B):
        pstart.append(P)
        if nchunks[b] > 1:
            P += nchunks[b]

    words_items = []
    indptr_w = [0]
    for w in range(W):
        for (b, k, _t) in lists[w]:
            begin = int(kv_indptr[b]) + k * c * T
            end = min(int(kv_indptr[b + 1]), begin + c * T)
            part = pstart[b] + k if nchunks[b] > 1 else -1
            words_items += [b, begin, end, part]
        indptr_w.append(len(words_items) // 4)
    n_items = len(words_items) // 4

    merge = []
    for b in range(B):
        if nchunks[b] != 1:
            p0 = pstart[b]
            p1 = p0 + (nchunks[b] if nchunks[b] > 1 else 0)
            merge += [b, p0, p1]
    n_merge = len(merge) // 3

    total_words = HEADER_WORDS + (W + 1) + 4 * n_items + 3 * n_merge
    header = [PLAN_MAGIC, PLAN_VERSION, B, H, variant, T, W, c, n_items, P, n_merge, 1, cpw,
              total_words, num_sms, 0]
    words = header + indptr_w + words_items + merge
    assert len(words) == total_words
    ws = WS_HEADER_BYTES + P * H * D_LATENT * 4 + P * H * 4
    ws = _ceil_div(ws, 256) * 256
    return words, ws
