"""fp64 CPU oracle for absorbed MLA decode.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA path (``mla_latent_kv_absorbed_gb300``) and imports nothing from it:
inputs arrive as plain numpy arrays (bf16 values as uint16 bit patterns) and are
widened to float64 exactly before any arithmetic.

What it computes (the plain definition; the kernel reaches the same result up
to rounding order):

  for request b and head h, with K_b = the cache rows named by
  kv_indices[kv_indptr[b]:kv_indptr[b+1]] (shape [L_b, 576]) and
  q = [q_nope[b,h], q_rope[b,h]] (576 wide):
      s_t  = sm_scale * (q_nope . c_t + q_rope . k_rope_t)           (dual-path score)
      lse  = ln sum_t exp(s_t)                                        (natural log, of the SCALED scores)
      out  = sum_t softmax(s)_t * c_t                                 (the latent is the value)

Sources, by page and section:
  * "实现差距：MLA 与 DeepSeek V3", section 2.4 "MLA Pallas Kernel (V2 生产版本)",
    core computation: the latent-path and rope-path dot products are added
    and the sum is multiplied by sm_scale (s_t above), an FA2-style online
    softmax follows, and the softmax weights multiply the latent rows, which
    serve as the values.  The oracle takes the softmax in one pass (max, then
    exp) instead of online.
  * same page, section 2.1 "Absorbed MLA 投影流程": kv_a_proj_with_mqa gives a
    576-wide row split as kv_latent (512) then k_rope (64) -- the row layout.
  * "Attention backends", paragraph "MLA": one 576-wide vector per token, 576
    wide for k and 512 for v, shared by all query heads.
  * "Attention backends", paragraph "FlashAttention": Flash-Decoding splits the
    keys across blocks and merges partial results with the same rescaling --
    ``merge_states``.
  * "MLA and torch.compile: v0.3's two sources", section "MLA: starting from a
    439-line commit": kv_b_proj split into w_kc and w_vc; decode multiplies
    q_nope by w_kc before attention and the latent output by w_vc after it --
    ``absorb_weights``, ``absorb_query``, ``project_output``,
    ``absorbed_attention``, ``decompressed_attention``.
  * same page, "Exercises", exercise 1: multiply-accumulate counts of the
    absorbing and decompressing paths -- ``mac_counts``.
  * "[sglang] EAGLE 트리 검증 어텐션 최적화", section "들어가며": draft tokens
    verified in one pass, each attending to the shared prefix and its
    ancestors -- ``decode_attention_multi_query`` (chain-shaped drafts),
    ``tree_ancestors`` and ``decode_attention_tree`` (topk > 1: a tree).
  * "MLA and torch.compile", section "MLA: starting from a 439-line commit"
    (FP8 KV cache; FP8 tensors are float8_e4m3fn) and "实现差距", section 2.4
    (FP8 packing of new rows) -- ``e4m3_to_f64``, ``f32_to_e4m3``,
    ``quantize_rows_e4m3``, ``decode_attention_fp8``, ``append_rows_fp8``.

Pins (tests/test_oracle_pins.py, CPU only): the absorption identity against a
decompressed multi-head attention evaluated with scipy's softmax; brute-force
closed forms for 1-3 tokens; split-and-merge equals the unsplit result;
invariance under relabelling cache slots; all-equal rows and q = 0 closed
forms; the MAC counts printed in exercise 1 (tests/golden/); the E4M3 code
table and rounding against torch's float8_e4m3fn conversions plus closed-form
codes, ties and saturation; FP8 decode against the bf16 decode of the same
(exactly representable) values; the draft tree against a brute-force masked
softmax whose visibility comes from a transitive closure of the parent
relation, against the chain and the star (every draft a child of the
context), a hand-made three-draft tree, and relabellings of sibling
subtrees.  Every function here is pinned by at least one of them.

Readings taken where the pages are silent: the rope key sits at columns
[512, 576) of a row; the LSE is natural-log and of the scaled scores; an empty
request gives out = 0 and lse = -inf; merging skips partials whose lse is -inf;
a slot named twice in one request counts twice; an FP8 cache holds E4M3
codes with one float32 scale for the whole cache; a draft tree lists its
drafts in generation order (a parent before its children, -1 for a child of
the verified context), and its drafts are the last W rows of the context.
"""
from __future__ import annotations

import numpy as np

KV_LORA_RANK = 512
QK_ROPE_HEAD_DIM = 64
KV_ROW = KV_LORA_RANK + QK_ROPE_HEAD_DIM


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def gather_rows(kv_cache_bits: np.ndarray, kv_indices: np.ndarray, begin: int, end: int) -> np.ndarray:
    """Rows kv_cache[kv_indices[begin:end]] as float64, shape [end-begin, 576].

    Page size 1: a request's cache is its list of slot numbers in token order
    ("Attention backends", paragraph "Paged, ragged batches").
    """
    idx = np.asarray(kv_indices[begin:end], dtype=np.int64)
    return bf16_bits_to_f64(kv_cache_bits[idx])


def partial_state(q_nope: np.ndarray, q_rope: np.ndarray, rows: np.ndarray, sm_scale: float):
    """Attention of one request's heads over a set of cache rows.

    q_nope [H,512], q_rope [H,64], rows [n,576] (all float64).
    Returns (o [H,512], lse [H]); o is already divided by the softmax sum.
    With n == 0: o = 0 and lse = -inf.
    """
    H = q_nope.shape[0]
    if rows.shape[0] == 0:
        return np.zeros((H, KV_LORA_RANK)), np.full(H, -np.inf)
    latent = rows[:, :KV_LORA_RANK]
    k_rope = rows[:, KV_LORA_RANK:]
    # dual-path score, scaled after the sum (section 2.4 of the sglang-jax gap page)
    s = (q_nope @ latent.T + q_rope @ k_rope.T) * sm_scale          # [H, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    denom = e.sum(axis=1, keepdims=True)
    lse = (m + np.log(denom))[:, 0]
    o = (e / denom) @ latent                                          # latent reused as value
    return o, lse


def decode_attention(q_nope_bits, q_rope_bits, kv_cache_bits, kv_indptr, kv_indices, sm_scale,
                     requests=None):
    """Absorbed MLA decode over a CSR batch.

    Returns (out [B,H,512], lse [B,H]) in float64.  With ``requests`` given,
    only those rows are computed; the others stay NaN.
    """
    qn = np.asarray(q_nope_bits)
    qr = np.asarray(q_rope_bits)
    B, H = qn.shape[0], qn.shape[1]
    out = np.full((B, H, KV_LORA_RANK), np.nan)
    lse = np.full((B, H), np.nan)
    todo = range(B) if requests is None else requests
    for b in todo:
        rows = gather_rows(kv_cache_bits, kv_indices, int(kv_indptr[b]), int(kv_indptr[b + 1]))
        o, l = partial_state(bf16_bits_to_f64(qn[b]), bf16_bits_to_f64(qr[b]), rows, sm_scale)
        out[b], lse[b] = o, l
    return out, lse


def decode_attention_multi_query(q_nope_bits, q_rope_bits, kv_cache_bits, kv_indptr, kv_indices, sm_scale, q_len):
    """Decode of q_len new tokens per request (speculative verification).

    q_nope [B, q_len, H, 512], q_rope [B, q_len, H, 64] (bf16 bits); request b's
    context of L_b rows ends with its q_len draft tokens, and query i
    (0 <= i < q_len) attends to the shared context and to its own ancestors,
    i.e. to the first L_b - q_len + i + 1 rows ("[sglang] EAGLE 트리 검증 어텐션
    최적화", section "들어가며": every query attends to the shared prefix and
    to its ancestor draft tokens; a chain of drafts is the causal case).
    Returns (out [B, q_len, H, 512], lse [B, q_len, H]).
    """
    qn = np.asarray(q_nope_bits)
    qr = np.asarray(q_rope_bits)
    B, Q, H = qn.shape[0], qn.shape[1], qn.shape[2]
    assert Q == q_len
    out = np.empty((B, Q, H, KV_LORA_RANK))
    lse = np.empty((B, Q, H))
    for b in range(B):
        lo, hi = int(kv_indptr[b]), int(kv_indptr[b + 1])
        assert hi - lo >= q_len, "a context holds at least its new tokens"
        for i in range(Q):
            rows = gather_rows(kv_cache_bits, kv_indices, lo, hi - q_len + i + 1)
            o, l = partial_state(bf16_bits_to_f64(qn[b, i]), bf16_bits_to_f64(qr[b, i]), rows, sm_scale)
            out[b, i], lse[b, i] = o, l
    return out, lse


def tree_ancestors(parents) -> list:
    """Ancestor-or-self sets of a draft tree.

    parents [W] (ints): parents[i] is the draft that draft i extends, or -1
    when it extends the verified context directly.  The drafts are listed in
    the order they were generated, so a parent comes before its children
    (parents[i] < i); anything else is rejected with ValueError.  Returns, for
    every i, the sorted list of i, its parent, its parent's parent, ... .
    ("[sglang] EAGLE 트리 검증 어텐션 최적화", section "들어가며": with topk > 1
    the drafts form a tree, and each query token attends only to its own
    ancestor chain among them.)
    """
    par = [int(x) for x in np.asarray(parents).reshape(-1)]
    out = []
    for i, pi in enumerate(par):
        if not -1 <= pi < i:
            raise ValueError(f"draft {i}: parent {pi} is not an earlier draft or -1")
        chain = [i] if pi < 0 else out[pi] + [i]
        out.append(sorted(chain))
    return out


def decode_attention_tree(q_nope_bits, q_rope_bits, kv_cache_bits, kv_indptr, kv_indices, sm_scale, parents):
    """Verification of a tree of W draft tokens per request in one pass.

    q_nope [B, W, H, 512], q_rope [B, W, H, 64] (bf16 bits); request b's
    context of L_b rows ends with its W drafts in their generation order,
    parents [B, W] as in ``tree_ancestors``.  Query i sees the first L_b - W
    rows (the verified context, shared by every draft) and, among the drafts,
    exactly its ancestors and itself ("[sglang] EAGLE 트리 검증 어텐션 최적화",
    section "들어가며").  A chain (parents[i] = i - 1) is
    ``decode_attention_multi_query``.  Returns (out [B, W, H, 512],
    lse [B, W, H]).
    """
    qn = np.asarray(q_nope_bits)
    qr = np.asarray(q_rope_bits)
    B, W, H = qn.shape[0], qn.shape[1], qn.shape[2]
    parents = np.asarray(parents).reshape(B, W)
    out = np.empty((B, W, H, KV_LORA_RANK))
    lse = np.empty((B, W, H))
    for b in range(B):
        lo, hi = int(kv_indptr[b]), int(kv_indptr[b + 1])
        if hi - lo < W:
            raise ValueError("a context holds at least its draft tokens")
        first = hi - W                                   # the first draft's position in kv_indices
        anc = tree_ancestors(parents[b])
        for i in range(W):
            slots = np.concatenate([np.asarray(kv_indices[lo:first], dtype=np.int64),
                                    np.asarray([kv_indices[first + a] for a in anc[i]], dtype=np.int64)])
            rows = bf16_bits_to_f64(kv_cache_bits[slots])
            o, l = partial_state(bf16_bits_to_f64(qn[b, i]), bf16_bits_to_f64(qr[b, i]), rows, sm_scale)
            out[b, i], lse[b, i] = o, l
    return out, lse


def merge_states(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Combine partial states of disjoint key sets by LSE rescaling.

    o_parts [P,H,512] (each already normalised), lse_parts [P,H].
      M = max_i lse_i;  w_i = exp(lse_i - M);
      out = sum_i w_i o_i / sum_i w_i;  lse = M + ln sum_i w_i.
    Partials with lse = -inf carry no weight; if every partial is empty the
    result is out = 0, lse = -inf.
    ("Attention backends", paragraph "FlashAttention": Flash-Decoding merges
    partial results with the same rescaling; the EAGLE tree-verify PR page
    merges prefix and suffix attention by LSE in its introduction.)
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    P, H = lse_parts.shape
    out = np.zeros((H, o_parts.shape[2]))
    lse = np.full(H, -np.inf)
    for h in range(H):
        l = lse_parts[:, h]
        live = np.isfinite(l)
        if not live.any():
            continue
        M = l[live].max()
        w = np.exp(l[live] - M)
        out[h] = (w[:, None] * o_parts[live, h, :]).sum(axis=0) / w.sum()
        lse[h] = M + np.log(w.sum())
    return out, lse


# ----------------------------------------------------------------------------
# Weight absorption: used only to pin the decode definition above against an
# ordinary multi-head attention over decompressed keys and values.
# ----------------------------------------------------------------------------

def absorb_weights(kv_b_proj: np.ndarray, qk_nope_head_dim: int, v_head_dim: int):
    """Split kv_b_proj [H*(nope+v), 512] into per-head w_kc and w_vc.

    Following "MLA and torch.compile: v0.3's two sources", section "MLA:
    starting from a 439-line commit": unflatten dim 0 to [H, nope+v, 512] and
    split along dim 1.  Returns
      w_kc [H, nope, 512]  (used as bmm(q_nope[H,B,nope], w_kc) -> [H,B,512])
      w_vc [H, 512, v]     (used as bmm(attn[H,B,512], w_vc)   -> [H,B,v])
    """
    rank = kv_b_proj.shape[1]
    w = kv_b_proj.reshape(-1, qk_nope_head_dim + v_head_dim, rank)
    w_kc = w[:, :qk_nope_head_dim, :]
    w_vc = np.transpose(w[:, qk_nope_head_dim:, :], (0, 2, 1))
    return w_kc, w_vc


def absorbed_attention(q_nope_heads, q_rope_heads, latents, k_rope, kv_b_proj, sm_scale,
                       qk_nope_head_dim, v_head_dim):
    """Decode for one request on the absorbing path, in float64.

    q_nope_heads [H, nope] (before absorption), q_rope_heads [H, 64],
    latents [L, 512], k_rope [L, 64].  q_nope is moved into the latent space by
    w_kc, attention runs on the latent rows (``partial_state``), and the latent
    output is moved to the value space by w_vc.  Returns [H, v].
    """
    w_kc, w_vc = absorb_weights(kv_b_proj, qk_nope_head_dim, v_head_dim)
    q_lat = absorb_query(q_nope_heads[None], w_kc)[0]                # bmm(q_nope, w_kc)
    rows = np.concatenate([latents, k_rope], axis=1)
    o_lat, _ = partial_state(q_lat, q_rope_heads, rows, sm_scale)
    return project_output(o_lat[None], w_vc)[0]                      # bmm(attn, w_vc)


def absorb_query(q_nope: np.ndarray, w_kc: np.ndarray) -> np.ndarray:
    """q_nope [B, H, nope] times each head's w_kc [H, nope, 512] -> [B, H, 512].

    The query-side bmm of the absorbing path ("MLA and torch.compile", section
    "MLA: starting from a 439-line commit": q_nope is multiplied by w_kc before
    attention).  Inputs as float64 (or bf16 bits widened by the caller).
    """
    return np.einsum("bhn,hnr->bhr", np.asarray(q_nope, np.float64), np.asarray(w_kc, np.float64))


def project_output(o_lat: np.ndarray, w_vc: np.ndarray) -> np.ndarray:
    """o_lat [B, H, 512] times each head's w_vc [H, 512, v] -> [B, H, v].

    The output-side bmm of the absorbing path (same section: the latent output
    of the attention is multiplied by w_vc).
    """
    return np.einsum("bhr,hrv->bhv", np.asarray(o_lat, np.float64), np.asarray(w_vc, np.float64))


def decompressed_attention(q_nope_heads, q_rope_heads, latents, k_rope, kv_b_proj, sm_scale,
                           qk_nope_head_dim, v_head_dim):
    """Decode for one request on the decompressing path, in float64.

    Every head gets its own keys k_{h,t} = [W_UK[h] c_t ; k_rope_t] and values
    v_{h,t} = W_UV[h] c_t, expanded from the latent rows with the kv_b_proj
    weights, and ordinary attention runs per head (scipy's softmax).  This is
    the path the absorbing one must equal ("MLA and torch.compile", self-test
    answer 2 and section "MLA: starting from a 439-line commit").  Returns [H, v].
    """
    from scipy.special import softmax

    H = q_nope_heads.shape[0]
    rank = kv_b_proj.shape[1]
    w = kv_b_proj.reshape(H, qk_nope_head_dim + v_head_dim, rank)
    out = np.empty((H, v_head_dim))
    for h in range(H):
        k_nope = latents @ w[h, :qk_nope_head_dim, :].T             # [L, nope]
        v = latents @ w[h, qk_nope_head_dim:, :].T                   # [L, v]
        keys = np.concatenate([k_nope, k_rope], axis=1)               # [L, nope+64]
        q = np.concatenate([q_nope_heads[h], q_rope_heads[h]])
        p = softmax(sm_scale * (keys @ q))
        out[h] = p @ v
    return out


def append_rows(kv_cache_bits: np.ndarray, slots: np.ndarray, rows_bits: np.ndarray) -> np.ndarray:
    """The cache after a decode step's append: row b (576 wide, latent then
    rope key) goes to slot slots[b]; every other row is unchanged.  Returns a
    new array ("实现差距：MLA 与 DeepSeek V3", section 2.4: the Pallas V2 kernel
    writes the new token's kv_c and k_pe into the cache pages before attending).
    Slots must be distinct and inside the pool."""
    out = np.array(kv_cache_bits, copy=True)
    idx = np.asarray(slots, dtype=np.int64)
    assert len(set(idx.tolist())) == idx.shape[0], "slots must be distinct"
    out[idx] = np.asarray(rows_bits)
    return out


# ------------------------------------------------------------ FP8 latent cache
# "MLA and torch.compile: v0.3's two sources", section "MLA: starting from a
# 439-line commit": an FP8 KV cache is one of the four parts of the 3-7x, and
# the same section's FP8 weights are torch.float8_e4m3fn; "实现差距：MLA 与
# DeepSeek V3", section 2.4: the V2 kernel packs new rows into an FP8 cache.
# Reading taken (the pages give no format or scale): the cache holds E4M3
# codes (the "fn" variant -- no infinities, largest finite 448), one byte per
# value, 576 per row; a row value is code value x kv_scale, one float32 scale
# for the whole cache.

E4M3_MAX = 448.0


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact value of E4M3 codes (uint8): sign bit 7, exponent bits 3-6 with
    bias 7, mantissa bits 0-2; exponent field 0 is subnormal (m/8 x 2^-6);
    0x7F and 0xFF are NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    return np.where((c & 0x7F) == 0x7F, np.nan, sign * mag)


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Round float32 values to E4M3 codes: to the nearest finite value, a tie
    to the code with an even last bit, magnitudes from 448 up (infinity too)
    to 448, NaN to 0x7F; the sign is kept (a value that rounds to zero gives
    +0 or -0).  Found by search over the 127 non-negative finite values."""
    xf = np.asarray(x, dtype=np.float32)
    a = np.abs(xf.astype(np.float64))
    grid = e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))          # codes 0..0x7E: 0 .. 448, increasing
    i = np.clip(np.searchsorted(grid, a, side="right") - 1, 0, 0x7E)
    j = np.minimum(i + 1, 0x7E)
    d_lo, d_hi = a - grid[i], grid[j] - a
    up = (j > i) & ((d_hi < d_lo) | ((d_hi == d_lo) & (i % 2 == 1)))
    code = np.where(up, j, i)
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    code = code | np.where(np.signbit(xf), 0x80, 0)
    return np.where(np.isnan(xf), 0x7F, code).astype(np.uint8)


def quantize_rows_e4m3(rows_bits: np.ndarray, kv_scale: float) -> np.ndarray:
    """FP8 codes of bf16 cache rows: each value divided by the cache scale in
    float32 (one IEEE division, correctly rounded), then rounded to E4M3."""
    x = bf16_bits_to_f64(rows_bits).astype(np.float32)             # exact
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        y = x / np.float32(kv_scale)
    return f32_to_e4m3(y)


def decode_attention_fp8(q_nope_bits, q_rope_bits, kv_codes, kv_scale, kv_indptr, kv_indices, sm_scale,
                         requests=None):
    """Absorbed MLA decode over an FP8 cache: every row value is its E4M3 code
    value times kv_scale (the float32 scale widened exactly); otherwise the
    same definition as ``decode_attention`` (the bf16 query is used as is)."""
    qn = np.asarray(q_nope_bits)
    qr = np.asarray(q_rope_bits)
    B, H = qn.shape[0], qn.shape[1]
    scale = float(np.float32(kv_scale))
    out = np.full((B, H, KV_LORA_RANK), np.nan)
    lse = np.full((B, H), np.nan)
    todo = range(B) if requests is None else requests
    for b in todo:
        idx = np.asarray(kv_indices[int(kv_indptr[b]):int(kv_indptr[b + 1])], dtype=np.int64)
        rows = e4m3_to_f64(np.asarray(kv_codes)[idx]) * scale
        o, l = partial_state(bf16_bits_to_f64(qn[b]), bf16_bits_to_f64(qr[b]), rows, sm_scale)
        out[b], lse[b] = o, l
    return out, lse


def append_rows_fp8(kv_codes: np.ndarray, slots: np.ndarray, rows_bits: np.ndarray, kv_scale: float) -> np.ndarray:
    """The FP8 cache after a decode step's append: slot slots[b] receives the
    codes of bf16 row b (``quantize_rows_e4m3``); every other row is unchanged."""
    out = np.array(kv_codes, copy=True)
    idx = np.asarray(slots, dtype=np.int64)
    assert len(set(idx.tolist())) == idx.shape[0], "slots must be distinct"
    out[idx] = quantize_rows_e4m3(rows_bits, kv_scale)
    return out


def mac_counts(num_heads: int, qk_nope_head_dim: int, kv_lora_rank: int, history: int):
    """Multiply-accumulates to bring one decode query against the history.

    Absorbing path: each head maps its q_nope (nope) through w_kc (nope x rank):
    H * nope * rank, independent of the history.  Decompressing path: every
    historical latent is mapped back to H heads of nope dims:
    history * rank * H * nope.  ("MLA and torch.compile", "Exercises", 1.)
    """
    absorbing = num_heads * qk_nope_head_dim * kv_lora_rank
    decompressing = history * kv_lora_rank * num_heads * qk_nope_head_dim
    return absorbing, decompressing
