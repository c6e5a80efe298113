"""Pins for the fp64 oracle: facts fixed by the pages and by the mathematics,
none of them a retyping of the oracle's own formula.  CPU only.

Each check is chosen so that a plausible mistake in the oracle (dropped rope
term, scale applied to one path only, wrong value columns, transposed operand,
log base, merge weight sign) fails at least one of them; the planted-mistake
tests at the bottom show that.
"""
import math
import os

import numpy as np
import pytest

from oracle import mla_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SM = 1.0 / math.sqrt(192.0)


def _rows(rng, n):
    return rng.standard_normal((n, 576))


def _dot(a, b):
    return math.fsum(float(x) * float(y) for x, y in zip(a, b))


def _score(qn, qr, row, scale):
    # plain python dual-path score, element by element
    return scale * (_dot(qn, row[:512]) + _dot(qr, row[512:]))


# --------------------------------------------------------------------------
# 1. absorption identity vs decompressed multi-head attention (scipy softmax)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("H,L", [(2, 1), (3, 5), (4, 17)])
def test_absorption_identity_matches_decompressed_mha(H, L):
    rng = np.random.default_rng(7 + H * 31 + L)
    nope, vdim = 128, 128
    kv_b_proj = rng.standard_normal((H * (nope + vdim), 512)) / math.sqrt(512)
    q_nope = rng.standard_normal((H, nope))
    q_rope = rng.standard_normal((H, 64))
    lat = rng.standard_normal((L, 512))
    k_rope = rng.standard_normal((L, 64))
    a = O.absorbed_attention(q_nope, q_rope, lat, k_rope, kv_b_proj, SM, nope, vdim)
    d = O.decompressed_attention(q_nope, q_rope, lat, k_rope, kv_b_proj, SM, nope, vdim)
    assert a.shape == (H, vdim)
    np.testing.assert_allclose(a, d, rtol=1e-11, atol=1e-12)


def test_absorb_query_and_project_output_are_per_head_products():
    # each head's rows are multiplied by that head's own matrix only: a head
    # or operand mix-up changes a brute-force dot product here
    rng = np.random.default_rng(11)
    B, H, n, r = 2, 3, 4, 5
    q = rng.standard_normal((B, H, n))
    w = rng.standard_normal((H, n, r))
    a = O.absorb_query(q, w)
    assert a.shape == (B, H, r)
    for b in range(B):
        for h in range(H):
            for j in range(r):
                assert abs(a[b, h, j] - sum(q[b, h, i] * w[h, i, j] for i in range(n))) < 1e-12
    o = rng.standard_normal((B, H, r))
    wv = rng.standard_normal((H, r, n))
    pr = O.project_output(o, wv)
    assert pr.shape == (B, H, n)
    for b in range(B):
        for h in range(H):
            for j in range(n):
                assert abs(pr[b, h, j] - sum(o[b, h, i] * wv[h, i, j] for i in range(r))) < 1e-12


def test_append_then_decode_equals_decode_over_the_extended_rows():
    # appending a request's new row to a free slot and adding that slot to its
    # index list is the same as attending over its old rows plus the new row
    rng = np.random.default_rng(21)
    pool, H, L = 40, 3, 6
    bits = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kv = bits(rng.standard_normal((pool, 576)))
    new = bits(rng.standard_normal((1, 576)))
    idx = rng.permutation(pool - 1)[:L].astype(np.int32)
    kv2 = O.append_rows(kv, np.array([pool - 1]), new)
    assert np.array_equal(kv2[:pool - 1], kv[:pool - 1]) and np.array_equal(kv2[pool - 1], new[0])
    qn, qr = bits(rng.standard_normal((1, H, 512))), bits(rng.standard_normal((1, H, 64)))
    ind2 = np.concatenate([idx, [pool - 1]]).astype(np.int32)
    o, l = O.decode_attention(qn, qr, kv2, np.array([0, L + 1]), ind2, SM)
    rows = np.concatenate([O.bf16_bits_to_f64(kv[idx]), O.bf16_bits_to_f64(new)], axis=0)
    ro, rl = O.partial_state(O.bf16_bits_to_f64(qn[0]), O.bf16_bits_to_f64(qr[0]), rows, SM)
    np.testing.assert_allclose(o[0], ro, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(l[0], rl, rtol=1e-13, atol=1e-13)


def test_multi_query_causal_decode_pins():
    # (a) q_len = 1 is the ordinary decode; (b) query i of a request equals an
    # ordinary decode of that request truncated to its causal length; (c) with
    # a single-row context extension, the last query's lse is the brute-force
    # log-sum-exp over every row
    rng = np.random.default_rng(33)
    bits = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    pool, H, Q = 50, 2, 3
    kv = bits(rng.standard_normal((pool, 576)))
    lens = [3, 7]
    ind = rng.permutation(pool)[:sum(lens)].astype(np.int32)
    ptr = np.array([0, 3, 10])
    qn1, qr1 = bits(rng.standard_normal((2, H, 512))), bits(rng.standard_normal((2, H, 64)))
    o1, l1 = O.decode_attention_multi_query(qn1[:, None], qr1[:, None], kv, ptr, ind, SM, 1)
    r1, rl1 = O.decode_attention(qn1, qr1, kv, ptr, ind, SM)
    np.testing.assert_array_equal(o1[:, 0], r1)
    np.testing.assert_array_equal(l1[:, 0], rl1)
    qn, qr = bits(rng.standard_normal((2, Q, H, 512))), bits(rng.standard_normal((2, Q, H, 64)))
    o, l = O.decode_attention_multi_query(qn, qr, kv, ptr, ind, SM, Q)
    for b in range(2):
        for i in range(Q):
            n = lens[b] - Q + i + 1
            tr_ptr = np.array([0, n])
            tr_ind = ind[ptr[b]:ptr[b] + n]
            ro, rl = O.decode_attention(qn[b, i][None], qr[b, i][None], kv, tr_ptr, tr_ind, SM)
            np.testing.assert_allclose(o[b, i], ro[0], rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(l[b, i], rl[0], rtol=1e-13, atol=1e-13)
    b, i, h = 1, Q - 1, 1
    q = np.concatenate([O.bf16_bits_to_f64(qn[b, i, h]), O.bf16_bits_to_f64(qr[b, i, h])])
    s_all = [SM * _dot(q, O.bf16_bits_to_f64(kv[ind[ptr[b] + t]])) for t in range(lens[b])]
    assert abs(l[b, i, h] - math.log(sum(math.exp(x) for x in s_all))) < 1e-12


def test_absorb_weights_layout():
    # kv_b_proj rows are [head][nope + v]; w_kc must pick the first nope rows
    # of each head's block, w_vc the remaining v rows, transposed.
    H, nope, vdim, R = 3, 4, 5, 6
    w = np.arange(H * (nope + vdim) * R, dtype=np.float64).reshape(H * (nope + vdim), R)
    w_kc, w_vc = O.absorb_weights(w, nope, vdim)
    assert w_kc.shape == (H, nope, R) and w_vc.shape == (H, R, vdim)
    for h in range(H):
        for i in range(nope):
            assert np.array_equal(w_kc[h, i], w[h * (nope + vdim) + i])
        for j in range(vdim):
            assert np.array_equal(w_vc[h, :, j], w[h * (nope + vdim) + nope + j])


# --------------------------------------------------------------------------
# 2. brute force on 1-3 tokens
# --------------------------------------------------------------------------

def test_one_token_closed_form():
    rng = np.random.default_rng(11)
    H = 3
    qn, qr, rows = rng.standard_normal((H, 512)), rng.standard_normal((H, 64)), _rows(rng, 1)
    o, lse = O.partial_state(qn, qr, rows, SM)
    for h in range(H):
        assert np.array_equal(o[h], rows[0, :512])          # softmax of one score is 1
        assert lse[h] == pytest.approx(_score(qn[h], qr[h], rows[0], SM), abs=1e-12)


def test_two_token_closed_form():
    rng = np.random.default_rng(12)
    H = 4
    qn, qr, rows = rng.standard_normal((H, 512)), rng.standard_normal((H, 64)), _rows(rng, 2)
    o, lse = O.partial_state(qn, qr, rows, SM)
    for h in range(H):
        s0 = _score(qn[h], qr[h], rows[0], SM)
        s1 = _score(qn[h], qr[h], rows[1], SM)
        p0 = 1.0 / (1.0 + math.exp(s1 - s0))
        want = p0 * rows[0, :512] + (1.0 - p0) * rows[1, :512]
        np.testing.assert_allclose(o[h], want, rtol=1e-12, atol=1e-13)
        assert lse[h] == pytest.approx(max(s0, s1) + math.log1p(math.exp(-abs(s1 - s0))), abs=1e-12)


def test_three_token_brute_force():
    rng = np.random.default_rng(13)
    H = 2
    qn, qr, rows = rng.standard_normal((H, 512)), rng.standard_normal((H, 64)), _rows(rng, 3)
    o, lse = O.partial_state(qn, qr, rows, SM)
    for h in range(H):
        s = [_score(qn[h], qr[h], rows[t], SM) for t in range(3)]
        e = [math.exp(x) for x in s]
        z = math.fsum(e)
        for d in range(0, 512, 37):
            want = math.fsum(e[t] / z * rows[t, d] for t in range(3))
            assert o[h, d] == pytest.approx(want, rel=1e-12, abs=1e-13)
        assert lse[h] == pytest.approx(math.log(z), abs=1e-12)


def test_scale_applies_to_both_paths():
    # with q_nope = 0 the score is sm_scale * rope part only; a scale applied to
    # one path only (or none) changes lse for a single token
    rng = np.random.default_rng(14)
    qr = rng.standard_normal((1, 64))
    rows = _rows(rng, 1)
    _, lse = O.partial_state(np.zeros((1, 512)), qr, rows, 0.25)
    assert lse[0] == pytest.approx(0.25 * _dot(qr[0], rows[0, 512:]), abs=1e-12)
    _, lse = O.partial_state(rng.standard_normal((1, 512)) * 0 + 1.0, np.zeros((1, 64)), rows, 0.5)
    assert lse[0] == pytest.approx(0.5 * math.fsum(rows[0, :512]), abs=1e-12)


# --------------------------------------------------------------------------
# 3. split-KV + LSE merge equals the unsplit result
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_split_merge_equals_unsplit(seed):
    rng = np.random.default_rng(100 + seed)
    H, L = 5, 97
    qn, qr, rows = rng.standard_normal((H, 512)), rng.standard_normal((H, 64)), _rows(rng, L) * 2.0
    ref_o, ref_l = O.partial_state(qn, qr, rows, SM)
    ncut = int(rng.integers(2, 6))
    cuts = sorted(set(int(c) for c in rng.integers(1, L, size=ncut)) | {0}) + [L]
    pieces, start = [], 0
    for c in cuts:
        pieces.append((start, c))        # may be empty
        start = c
    parts = [O.partial_state(qn, qr, rows[a:b], SM) for a, b in pieces]
    o, l = O.merge_states(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(o, ref_o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)


def test_merge_all_empty_and_single():
    o, l = O.merge_states(np.zeros((2, 3, 512)), np.full((2, 3), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(l))
    rng = np.random.default_rng(5)
    x = rng.standard_normal((1, 3, 512))
    lx = rng.standard_normal((1, 3))
    o, l = O.merge_states(x, lx)
    np.testing.assert_allclose(o, x[0], rtol=1e-15)
    np.testing.assert_allclose(l, lx[0], rtol=1e-15)


def test_empty_request():
    o, l = O.partial_state(np.ones((2, 512)), np.ones((2, 64)), np.zeros((0, 576)), SM)
    assert np.all(o == 0) and np.all(np.isneginf(l))


# --------------------------------------------------------------------------
# 4. relabelling the physical slots changes nothing (bit for bit)
# --------------------------------------------------------------------------

def test_slot_permutation_invariance():
    from mla_latent_kv_absorbed_gb300 import workloads as W
    bt = W.make_batch([3, 0, 40, 129], heads=16, pool=300, seed=3)
    out1, lse1 = O.decode_attention(bt.q_nope, bt.q_rope, bt.kv_cache, bt.kv_indptr, bt.kv_indices, SM)
    perm = np.random.default_rng(9).permutation(bt.pool)
    kv2 = np.empty_like(bt.kv_cache)
    kv2[perm] = bt.kv_cache                      # kv'[pi(s)] = kv[s]
    idx2 = perm[bt.kv_indices].astype(np.int32)  # indices' = pi(indices)
    out2, lse2 = O.decode_attention(bt.q_nope, bt.q_rope, kv2, bt.kv_indptr, idx2, SM)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


# --------------------------------------------------------------------------
# 5. closed forms
# --------------------------------------------------------------------------

def test_all_rows_equal():
    rng = np.random.default_rng(21)
    H, L = 3, 50
    row = rng.standard_normal(576)
    rows = np.tile(row, (L, 1))
    qn, qr = rng.standard_normal((H, 512)), rng.standard_normal((H, 64))
    o, lse = O.partial_state(qn, qr, rows, SM)
    for h in range(H):
        np.testing.assert_allclose(o[h], row[:512], rtol=1e-13)
        assert lse[h] == pytest.approx(_score(qn[h], qr[h], row, SM) + math.log(L), abs=1e-11)


def test_zero_query_is_uniform_mean():
    rng = np.random.default_rng(22)
    L = 33
    rows = _rows(rng, L)
    o, lse = O.partial_state(np.zeros((2, 512)), np.zeros((2, 64)), rows, SM)
    for h in range(2):
        want = [math.fsum(rows[:, d]) / L for d in range(512)]
        np.testing.assert_allclose(o[h], want, rtol=1e-12, atol=1e-14)
        assert lse[h] == pytest.approx(math.log(L), abs=1e-13)


def test_bf16_widening_is_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x3F81, 0x7F7F, 0x0001, 0x4049], dtype=np.uint16)
    want = [1.0, -1.0, 0.0, -0.0, 1.0 + 2.0 ** -7, (2 - 2.0 ** -7) * 2.0 ** 127, 2.0 ** -133, 3.140625]
    got = O.bf16_bits_to_f64(bits)
    assert [float(x) for x in got] == want


def test_mac_counts_golden():
    with open(os.path.join(GOLDEN, "mac_counts.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for H, nope, rank, hist, absorb, decomp, p_abs, p_dec in rows:
        a, d = O.mac_counts(int(H), int(nope), int(rank), int(hist))
        assert (a, d) == (int(absorb), int(decomp))
        assert round(a / 1e6, 1) == float(p_abs.rstrip("M"))        # "~8.4M"
        assert round(d / 1e9) == int(p_dec.rstrip("G"))              # "~34G"


def test_row_width_golden():
    with open(os.path.join(GOLDEN, "row_widths.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for rank, rope, width, mha, padded, ratio in rows:
        assert O.KV_LORA_RANK == int(rank) and O.QK_ROPE_HEAD_DIM == int(rope)
        assert O.KV_ROW == int(width)
        assert 128 * 128 * 2 == int(mha)
        assert round(int(mha) / int(padded)) == int(ratio)


# --------------------------------------------------------------------------
# planted mistakes: each plausible oracle bug is caught by some pin above
# --------------------------------------------------------------------------

def _mutant_partial(kind):
    def f(q_nope, q_rope, rows, sm_scale):
        H = q_nope.shape[0]
        if rows.shape[0] == 0:
            return np.zeros((H, 512)), np.full(H, -np.inf)
        lat, kr = rows[:, :512], rows[:, 512:]
        if kind == "drop_rope":
            s = (q_nope @ lat.T) * sm_scale
        elif kind == "scale_nope_only":
            s = q_nope @ lat.T * sm_scale + q_rope @ kr.T
        elif kind == "value_offset":
            lat_v = rows[:, 64:]
            s = (q_nope @ lat.T + q_rope @ kr.T) * sm_scale
            m = s.max(1, keepdims=True); e = np.exp(s - m); z = e.sum(1, keepdims=True)
            return (e / z) @ lat_v, (m + np.log(z))[:, 0]
        elif kind == "log2_lse":
            s = (q_nope @ lat.T + q_rope @ kr.T) * sm_scale
            m = s.max(1, keepdims=True); e = np.exp(s - m); z = e.sum(1, keepdims=True)
            return (e / z) @ lat, (m + np.log2(z))[:, 0]
        else:
            raise ValueError(kind)
        m = s.max(1, keepdims=True); e = np.exp(s - m); z = e.sum(1, keepdims=True)
        return (e / z) @ lat, (m + np.log(z))[:, 0]
    return f


PIN_TESTS = [
    lambda: test_absorption_identity_matches_decompressed_mha(3, 5),
    test_one_token_closed_form, test_two_token_closed_form, test_three_token_brute_force,
    test_scale_applies_to_both_paths, test_all_rows_equal, test_zero_query_is_uniform_mean,
]


@pytest.mark.parametrize("kind", ["drop_rope", "scale_nope_only", "value_offset", "log2_lse"])
def test_planted_partial_mistakes_are_caught(kind, monkeypatch):
    monkeypatch.setattr(O, "partial_state", _mutant_partial(kind))
    failures = 0
    for t in PIN_TESTS:
        try:
            t()
        except AssertionError:
            failures += 1
    assert failures >= 1, f"mutant {kind} passed every pin"


def test_planted_merge_mistake_is_caught(monkeypatch):
    real = O.merge_states

    def bad(o_parts, lse_parts):       # weights exp(M - lse) instead of exp(lse - M)
        o_parts = np.asarray(o_parts); lse_parts = np.asarray(lse_parts)
        M = np.max(np.where(np.isfinite(lse_parts), lse_parts, -1e300), axis=0)
        w = np.where(np.isfinite(lse_parts), np.exp(M - lse_parts), 0.0)
        return (w[..., None] * o_parts).sum(0) / w.sum(0)[:, None], M + np.log(w.sum(0))

    monkeypatch.setattr(O, "merge_states", bad)
    for seed in range(3):
        with pytest.raises(AssertionError):
            test_split_merge_equals_unsplit(seed)
    monkeypatch.setattr(O, "merge_states", real)


# ------------------------------------------------------------ FP8 latent cache

def _torch_e4m3_values(codes):
    import torch
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def test_e4m3_code_table_matches_torch_and_closed_forms():
    pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    v, t = O.e4m3_to_f64(codes), _torch_e4m3_values(codes)
    assert np.array_equal(np.isnan(v), np.isnan(t)) and np.isnan(v).sum() == 2
    assert np.array_equal(v[~np.isnan(v)], t[~np.isnan(t)])
    # closed forms of the format: smallest subnormal, largest subnormal, smallest normal, one, largest finite
    for code, val in ((0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x38, 1.0), (0x7E, 448.0),
                      (0xFE, -448.0), (0x80, 0.0)):
        assert O.e4m3_to_f64(np.array([code], np.uint8))[0] == val


def test_e4m3_rounding_matches_torch_in_range():
    pytest.importorskip("torch")
    import torch
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(100000) * np.exp2(rng.uniform(-14, 9, 100000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.f32_to_e4m3(x), want)


def test_e4m3_ties_go_to_the_even_code_and_large_values_saturate():
    grid = O.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)       # every midpoint is exact in float32
    assert np.array_equal(mids.astype(np.float64), (grid[:-1] + grid[1:]) / 2)
    lo = np.arange(0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(O.f32_to_e4m3(mids), want.astype(np.uint8))
    assert np.array_equal(O.f32_to_e4m3(-mids), (want | 0x80).astype(np.uint8))
    big = np.array([448.0, 449.0, 463.9, 464.0, 1e6, np.inf, -1e30, -np.inf], np.float32)
    assert np.array_equal(O.f32_to_e4m3(big), np.array([0x7E] * 6 + [0xFE] * 2, np.uint8))
    assert O.f32_to_e4m3(np.array([np.nan], np.float32))[0] == 0x7F
    # below half the smallest subnormal: signed zero; just above: the smallest subnormal
    tiny = np.array([2.0 ** -11, -2.0 ** -11, 2.0 ** -10, 2.0 ** -10 * 1.0001], np.float32)
    assert np.array_equal(O.f32_to_e4m3(tiny), np.array([0x00, 0x80, 0x00, 0x01], np.uint8))
    # every finite code survives a round trip
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(O.f32_to_e4m3(O.e4m3_to_f64(codes).astype(np.float32)), codes)


def test_quantize_rows_divides_by_the_scale_then_rounds():
    from mla_latent_kv_absorbed_gb300 import workloads as W
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 256, size=(6, 576)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x42
    for scale in (1.0, 2.0 ** -5, 8.0):
        vals = O.e4m3_to_f64(codes) * scale                       # exact in bf16 for these scales
        bits = W.f32_to_bf16_bits(vals.astype(np.float32))
        assert np.array_equal(O.bf16_bits_to_f64(bits), vals)
        assert np.array_equal(O.quantize_rows_e4m3(bits, scale), codes)
    # the rounding sees the quotient: 1.0625 / 0.5 = 2.125 and 1.1875 / 0.5 = 2.375 are ties between codes
    # 0x40 = 2.0 / 0x41 = 2.25 and 0x41 / 0x42 = 2.5, so both go to the even code; 1.125 / 0.5 = 2.25 is exact
    one = W.f32_to_bf16_bits(np.array([1.0625, 1.1875, 1.125], np.float32))
    assert np.array_equal(O.quantize_rows_e4m3(one, 0.5), np.array([0x40, 0x42, 0x41], np.uint8))


def test_fp8_decode_equals_bf16_decode_of_the_same_values():
    from mla_latent_kv_absorbed_gb300 import workloads as W
    rng = np.random.default_rng(10)
    pool, H = 300, 4
    codes = O.f32_to_e4m3((rng.standard_normal((pool, 576)) * 16).astype(np.float32))
    lengths = [0, 1, 7, 120]
    indptr = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    indices = rng.permutation(pool)[:indptr[-1]].astype(np.int32)
    qn = W.f32_to_bf16_bits(rng.standard_normal((4, H, 512)).astype(np.float32))
    qr = W.f32_to_bf16_bits(rng.standard_normal((4, H, 64)).astype(np.float32))
    for scale in (1.0, 2.0 ** -5):
        bits = W.f32_to_bf16_bits((O.e4m3_to_f64(codes) * scale).astype(np.float32))
        ro, rl = O.decode_attention(qn, qr, bits, indptr, indices, SM)
        fo, fl = O.decode_attention_fp8(qn, qr, codes, scale, indptr, indices, SM)
        assert np.array_equal(ro, fo) and np.array_equal(rl, fl)
    # a scale is not a no-op: doubling it changes the scores
    fo2, _ = O.decode_attention_fp8(qn, qr, codes, 2.0 ** -4, indptr, indices, SM)
    assert not np.allclose(fo2[3], fo[3])


def test_fp8_append_touches_only_its_slots():
    from mla_latent_kv_absorbed_gb300 import workloads as W
    rng = np.random.default_rng(11)
    cache = rng.integers(0, 0x7E, size=(50, 576)).astype(np.uint8)
    rows = W.f32_to_bf16_bits(rng.standard_normal((3, 576)).astype(np.float32))
    slots = np.array([4, 17, 0], np.int32)
    after = O.append_rows_fp8(cache, slots, rows, 2.0 ** -5)
    keep = np.setdiff1d(np.arange(50), slots)
    assert np.array_equal(after[keep], cache[keep])
    assert np.array_equal(after[slots], O.quantize_rows_e4m3(rows, 2.0 ** -5))
    back = O.e4m3_to_f64(after[slots]) * 2.0 ** -5
    assert np.all(np.abs(back - O.bf16_bits_to_f64(rows)) <= np.abs(O.bf16_bits_to_f64(rows)) / 16 + 2.0 ** -15)
