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
  * loads are counted in tokens: a work item of n tokens costs its tiles,
    ceil(n / T) * T, plus the variant's ITEM_OVERHEAD (32 tokens for swab,
    256 for pair: a cost-model figure, measured per kernel); total = sum over
    requests of ceil(L_b / T) * T;
  * wrap-around fill: requests are walked in b order and poured into workers
    0, 1, ... in turn, each worker up to a load budget cap; a request is cut
    only where a worker is full, at a tile boundary of the request (so only
    its last piece can be ragged), and there are at most W - 1 cuts;
  * no cut piece is shorter than MIN_PIECE tokens and no worker's load
    exceeds cap: where the tail after the whole tiles that fit would be
    shorter than MIN_PIECE, the cut moves one tile earlier (the tail piece
    then holds a whole tile besides its ragged one); with less space than
    that the worker is closed;
  * cap starts at ceil((total + (nonempty + W - 1) * overhead) / W) and
    grows by CAP_STEP tokens until the fill fits on the W workers;
  * partial slots are numbered over the cut requests in (b, piece) order; an
    uncut request's item writes out/lse directly (partial = -1);
  * the merge list holds every request that is cut or empty, in b order, with
    its partial range (empty requests get an empty range).

Plan words (int32): a 16-word header, worker_indptr[W+1], 4 words per item
(b, kv_begin, kv_end, partial) grouped by worker in placement order, then 3
words per merge entry (b, p_begin, p_end).
"""
from __future__ import annotations

PLAN_MAGIC = 0x4D4C4131
PLAN_VERSION = 1
HEADER_WORDS = 16
MIN_PIECE = 64        # tokens
CAP_STEP = 8          # tokens
WS_HEADER_BYTES = 256
D_LATENT = 512

VARIANT_SWAB = 1
VARIANT_PAIR = 2
ITEM_OVERHEAD = {VARIANT_SWAB: 32, VARIANT_PAIR: 256}   # tokens per work item


def variant_for_heads(H: int):
    """(variant, tile_tokens, ctas_per_worker) or None when H is unsupported."""
    if H in (16, 32):
        return VARIANT_SWAB, 64, 1
    if 48 <= H <= 128 and H % 16 == 0:
        return VARIANT_PAIR, 64, 2
    return None


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


TILE = 64


def _round_up(n: int) -> int:
    return _ceil_div(n, TILE) * TILE


def _fill(lengths, W, cap, overhead):
    """Wrap-around fill with load budget cap: per-worker lists of
    (b, first token, tokens), or None when W workers do not suffice."""
    lists = [[] for _ in range(W)]
    w, used = 0, 0
    for b, t in enumerate(lengths):
        k0 = 0
        while k0 < t:
            if w == W:
                return None
            rem = t - k0
            space = cap - used - overhead
            fit = (space // TILE) * TILE if space > 0 else 0      # whole tiles that fit
            if _round_up(rem) <= space:
                take = rem
            elif fit >= MIN_PIECE and rem - fit >= MIN_PIECE:
                take = fit
            elif fit - TILE >= MIN_PIECE:
                take = fit - TILE                                  # the tail keeps a whole tile
            else:
                w, used = w + 1, 0
                continue
            lists[w].append((b, k0, take))
            used += _round_up(take) + overhead
            k0 += take
    return lists


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
    total = sum(_round_up(L) for L in lengths)
    nonempty = sum(1 for L in lengths if L > 0)

    overhead = ITEM_OVERHEAD[variant]
    if total > 0:
        cap = _ceil_div(total + (nonempty + W - 1) * overhead, W)
        while True:
            lists = _fill(lengths, W, cap, overhead)
            if lists is not None:
                break
            cap += CAP_STEP
    else:
        cap, lists = 0, [[] for _ in range(W)]

    npieces = [0] * B
    for lst in lists:
        for (b, _k0, _t) in lst:
            npieces[b] += 1
    pstart = []
    P = 0
    for b in range(B):
        pstart.append(P)
        if npieces[b] > 1:
            P += npieces[b]

    words_items = []
    indptr_w = [0]
    seen = [0] * B
    for w in range(W):
        for (b, k0, t) in lists[w]:
            begin = int(kv_indptr[b]) + k0
            end = begin + t
            part = pstart[b] + seen[b] if npieces[b] > 1 else -1
            seen[b] += 1
            words_items += [b, begin, end, part]
        indptr_w.append(len(words_items) // 4)
    n_items = len(words_items) // 4

    merge = []
    for b in range(B):
        if npieces[b] != 1:
            p0 = pstart[b]
            p1 = p0 + (npieces[b] if npieces[b] > 1 else 0)
            merge += [b, p0, p1]
    n_merge = len(merge) // 3

    total_words = HEADER_WORDS + (W + 1) + 4 * n_items + 3 * n_merge
    header = [PLAN_MAGIC, PLAN_VERSION, B, H, variant, T, W, cap, n_items, P, n_merge, 1, cpw,
              total_words, num_sms, 0]
    words = header + indptr_w + words_items + merge
    assert len(words) == total_words
    ws = WS_HEADER_BYTES + P * H * D_LATENT * 4 + P * H * 4
    ws = _ceil_div(ws, 256) * 256
    return words, ws
