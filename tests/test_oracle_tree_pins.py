"""Pins of the oracle's draft-tree verification (CPU only).

"[sglang] EAGLE 트리 검증 어텐션 최적화", section "들어가며": with topk > 1 the
draft tokens form a tree, the target model verifies the whole tree in one
pass, and each query token attends to the shared context and to its own
ancestor chain among the drafts.  ``decode_attention_tree`` is checked here
against a brute-force masked softmax whose visibility matrix comes from a
transitive closure of the parent relation (not from ``tree_ancestors``),
against the chain (the causal multi-query decode) and the star (every draft a
direct child of the context: one ordinary decode per draft), a three-draft
tree written out by hand, and a relabelling of sibling subtrees.
"""
import math

import numpy as np
import pytest

from oracle import mla_oracle as O

SM = 1.0 / math.sqrt(192.0)


def _bits(a):
    return (np.asarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _case(rng, lens, W, H, pool=None):
    pool = pool or sum(lens) + 7
    kv = _bits(rng.standard_normal((pool, 576)))
    ind = rng.permutation(pool)[:sum(lens)].astype(np.int32)
    ptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    qn = _bits(rng.standard_normal((len(lens), W, H, 512)))
    qr = _bits(rng.standard_normal((len(lens), W, H, 64)))
    return kv, ind, ptr, qn, qr


def _random_tree(rng, W):
    return np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, W)], dtype=np.int64)


def _closure(parents):
    """reach[i, j]: draft j is draft i or one of its ancestors, by iterating
    reach <- reach | reach . A (A[i, j] = draft j is the parent of draft i)
    until nothing changes."""
    W = len(parents)
    A = np.zeros((W, W), dtype=bool)
    for i, p in enumerate(parents):
        if p >= 0:
            A[i, p] = True
    reach = np.eye(W, dtype=bool)
    while True:
        nxt = reach | ((reach.astype(np.int64) @ A.astype(np.int64)) > 0)
        if np.array_equal(nxt, reach):
            return reach
        reach = nxt


def _brute(kv, ind, ptr, qn, qr, parents):
    """Masked softmax over every row of the context, element by element."""
    B, W, H = qn.shape[:3]
    out = np.empty((B, W, H, 512))
    lse = np.empty((B, W, H))
    for b in range(B):
        lo, hi = int(ptr[b]), int(ptr[b + 1])
        reach = _closure(parents[b])
        rows = O.bf16_bits_to_f64(kv[ind[lo:hi].astype(np.int64)])
        L = hi - lo
        for i in range(W):
            visible = [t for t in range(L) if t < L - W or reach[i, t - (L - W)]]
            for h in range(H):
                q = np.concatenate([O.bf16_bits_to_f64(qn[b, i, h]), O.bf16_bits_to_f64(qr[b, i, h])])
                s = [SM * math.fsum(q * rows[t]) for t in visible]
                m = max(s)
                w = [math.exp(x - m) for x in s]
                den = math.fsum(w)
                lse[b, i, h] = m + math.log(den)
                out[b, i, h] = sum(wk * rows[t, :512] for wk, t in zip(w, visible)) / den
    return out, lse


def test_ancestors_of_a_small_tree_and_invalid_parents():
    assert O.tree_ancestors([-1, 0, 0, 1, 3]) == [[0], [0, 1], [0, 2], [0, 1, 3], [0, 1, 3, 4]]
    assert O.tree_ancestors([-1, -1, 1]) == [[0], [1], [1, 2]]
    for bad in ([0], [-1, 1], [-1, 2, 0], [-2]):
        with pytest.raises(ValueError):
            O.tree_ancestors(bad)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tree_matches_brute_force_masked_softmax(seed):
    rng = np.random.default_rng(700 + seed)
    W, H = 6, 2
    lens = [W, W + 3, W + 11]               # the first request: drafts only, no shared context
    kv, ind, ptr, qn, qr = _case(rng, lens, W, H)
    parents = np.stack([_random_tree(rng, W) for _ in lens])
    o, l = O.decode_attention_tree(qn, qr, kv, ptr, ind, SM, parents)
    bo, bl = _brute(kv, ind, ptr, qn, qr, parents)
    np.testing.assert_allclose(o, bo, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l, bl, rtol=1e-12, atol=1e-12)


def test_chain_tree_is_the_causal_multi_query_decode():
    rng = np.random.default_rng(710)
    W, H = 4, 3
    kv, ind, ptr, qn, qr = _case(rng, [9, 4, 30], W, H)
    chain = np.tile(np.arange(-1, W - 1), (3, 1))
    o, l = O.decode_attention_tree(qn, qr, kv, ptr, ind, SM, chain)
    mo, ml = O.decode_attention_multi_query(qn, qr, kv, ptr, ind, SM, W)
    np.testing.assert_allclose(o, mo, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(l, ml, rtol=1e-13, atol=1e-13)


def test_star_tree_is_one_decode_per_draft_over_context_and_itself():
    rng = np.random.default_rng(720)
    W, H = 5, 2
    lens = [12, 5]
    kv, ind, ptr, qn, qr = _case(rng, lens, W, H)
    star = np.full((2, W), -1)
    o, l = O.decode_attention_tree(qn, qr, kv, ptr, ind, SM, star)
    for b, L in enumerate(lens):
        lo = int(ptr[b])
        for i in range(W):
            sub = np.concatenate([ind[lo:lo + L - W], [ind[lo + L - W + i]]])
            ro, rl = O.decode_attention(qn[b, i][None], qr[b, i][None], kv, np.array([0, len(sub)]), sub, SM)
            np.testing.assert_allclose(o[b, i], ro[0], rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(l[b, i], rl[0], rtol=1e-13, atol=1e-13)


def test_three_draft_tree_by_hand():
    # drafts: 0 extends the context, 1 and 2 both extend 0 (top-2 at the
    # second step); draft 2 must not see draft 1
    rng = np.random.default_rng(730)
    H = 1
    kv, ind, ptr, qn, qr = _case(rng, [5], 3, H)
    o, l = O.decode_attention_tree(qn, qr, kv, ptr, ind, SM, np.array([[-1, 0, 0]]))
    seen = {0: [0, 1, 2], 1: [0, 1, 2, 3], 2: [0, 1, 2, 4]}    # positions in the 5-row context
    for i, pos in seen.items():
        sub = ind[pos]
        ro, rl = O.decode_attention(qn[0, i][None], qr[0, i][None], kv, np.array([0, len(sub)]), sub, SM)
        np.testing.assert_allclose(o[0, i], ro[0], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(l[0, i], rl[0], rtol=1e-13, atol=1e-13)
    # and draft 2's result differs from what it would be if it saw draft 1
    wrong, _ = O.decode_attention(qn[0, 2][None], qr[0, 2][None], kv, np.array([0, 4]), ind[[0, 1, 2, 3]], SM)
    assert np.abs(o[0, 2] - wrong[0]).max() > 1e-3


def test_relabelling_sibling_subtrees_permutes_the_results():
    # old tree: 1 and 2 extend 0; 3 and 4 extend 1; 5 extends 2.  Listing the
    # subtree of 2 first gives the same tree under pi = old -> new index.
    rng = np.random.default_rng(740)
    W, H = 6, 2
    kv, ind, ptr, qn, qr = _case(rng, [W + 6], W, H)
    old = np.array([-1, 0, 0, 1, 1, 2])
    pi = np.array([0, 2, 1, 4, 5, 3])
    new = np.empty(W, dtype=np.int64)
    for o_, p_ in enumerate(old):
        new[pi[o_]] = -1 if p_ < 0 else pi[p_]
    assert list(new) == [-1, 0, 0, 1, 2, 2]
    first = int(ptr[1]) - W
    ind2 = ind.copy()
    qn2, qr2 = qn.copy(), qr.copy()
    for o_ in range(W):
        ind2[first + pi[o_]] = ind[first + o_]
        qn2[0, pi[o_]] = qn[0, o_]
        qr2[0, pi[o_]] = qr[0, o_]
    oa, la = O.decode_attention_tree(qn, qr, kv, ptr, ind, SM, old[None])
    ob, lb = O.decode_attention_tree(qn2, qr2, kv, ptr, ind2, SM, new[None])
    for o_ in range(W):
        np.testing.assert_allclose(ob[0, pi[o_]], oa[0, o_], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lb[0, pi[o_]], la[0, o_], rtol=1e-13, atol=1e-13)


def test_a_context_shorter_than_its_drafts_is_rejected():
    rng = np.random.default_rng(750)
    kv, ind, ptr, qn, qr = _case(rng, [2], 3, 1)
    with pytest.raises(ValueError):
        O.decode_attention_tree(qn, qr, kv, ptr, ind, SM, np.array([[-1, 0, 1]]))


@pytest.mark.parametrize("kind", ["no_self", "siblings_visible"])
def test_planted_ancestor_mistakes_are_caught(kind, monkeypatch):
    # a plausible slip in the ancestor sets must fail the brute-force pin
    real = O.tree_ancestors

    def wrong(parents):
        anc = real(parents)
        if kind == "no_self":
            return [a[:-1] if len(a) > 1 else a for a in anc]
        par = [int(x) for x in np.asarray(parents).reshape(-1)]
        return [sorted(set(a) | {j for j, pj in enumerate(par) if pj == par[i] and j != i}) for i, a in enumerate(anc)]

    rng = np.random.default_rng(760)
    W, H = 5, 1
    kv, ind, ptr, qn, qr = _case(rng, [W + 4], W, H)
    parents = np.array([[-1, 0, 0, 1, 1]])
    bo, bl = _brute(kv, ind, ptr, qn, qr, parents)
    monkeypatch.setattr(O, "tree_ancestors", wrong)
    o, l = O.decode_attention_tree(qn, qr, kv, ptr, ind, SM, parents)
    assert np.abs(o - bo).max() > 1e-6 or np.abs(l - bl).max() > 1e-6
