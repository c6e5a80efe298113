"""Properties of the split-KV plan restatement (oracle/plan_ref.py), CPU only.

The pages fix no chunking rule, only its job (cover every key once, balance
long and short contexts across SMs), so these pins check that job: exact
coverage, partial numbering, the merge list, and the wrap-around fill's
bounds (in tokens, pieces costed in whole tiles): no worker's load above the
budget cap, cap within 2 MIN_PIECE + CAP_STEP of the ideal
ceil((total + items) / W), cuts only at tile boundaries of the request, no
cut piece shorter than MIN_PIECE, and at most W - 1 cuts.
"""
import numpy as np
import pytest

from oracle import plan_ref as PR


def _decode(words):
    h = words[:16]
    assert h[0] == PR.PLAN_MAGIC and h[1] == PR.PLAN_VERSION
    B, H, variant, T, W, c, n, P, nm = h[2], h[3], h[4], h[5], h[6], h[7], h[8], h[9], h[10]
    off = 16
    wptr = words[off:off + W + 1]
    off += W + 1
    items = [tuple(words[off + 4 * i: off + 4 * i + 4]) for i in range(n)]
    off += 4 * n
    merge = [tuple(words[off + 3 * i: off + 3 * i + 3]) for i in range(nm)]
    off += 3 * nm
    assert off == len(words) == h[13]
    return dict(B=B, H=H, variant=variant, T=T, W=W, c=c, n=n, P=P, wptr=wptr, items=items, merge=merge)


def _check(indptr, H, sms):
    words, ws = PR.build_plan(indptr, H, sms)
    d = _decode(words)
    B = len(indptr) - 1
    T, c = d["T"], d["c"]
    assert d["wptr"][0] == 0 and d["wptr"][-1] == d["n"]
    assert all(a <= b for a, b in zip(d["wptr"], d["wptr"][1:]))
    ov = PR.ITEM_OVERHEAD[d["variant"]]
    items_max = c - ov if c else 0                 # tokens
    # exact coverage of each request's keys
    cover = {b: [] for b in range(B)}
    parts = {}
    for (b, s, e, p) in d["items"]:
        assert indptr[b] <= s < e <= indptr[b + 1]
        assert e - s <= items_max
        cover[b].append((s, e))
        if p >= 0:
            assert p not in parts
            parts[p] = (b, s)
    for b in range(B):
        segs = sorted(cover[b])
        pos = indptr[b]
        for s, e in segs:
            assert s == pos
            pos = e
        assert pos == indptr[b + 1]
    # partials: numbered over cut requests in (b, chunk) order
    assert sorted(parts) == list(range(d["P"]))
    order = sorted(parts.items(), key=lambda kv: kv[0])
    assert [bs for _, bs in order] == sorted(bs for _, bs in order)
    # merge list: every cut or empty request, with its partial range
    mset = {m[0]: m for m in d["merge"]}
    for b in range(B):
        nb = len(cover[b])
        if nb == 1:
            assert b not in mset
            assert all(p < 0 for (bb, _, _, p) in d["items"] if bb == b)
        else:
            _, p0, p1 = mset[b]
            assert p1 - p0 == (nb if nb > 1 else 0)
            assert sorted(p for (bb, _, _, p) in d["items"] if bb == b) == list(range(p0, p1))
    # fill bounds (tokens)
    lengths = [int(indptr[b + 1] - indptr[b]) for b in range(B)]
    rup = lambda n: -(-n // T) * T
    total, nonempty = sum(rup(L) for L in lengths), sum(1 for L in lengths if L > 0)
    loads = []
    for w in range(d["W"]):
        its = d["items"][d["wptr"][w]:d["wptr"][w + 1]]
        loads.append(sum(rup(e - s) + ov for (_, s, e, _) in its))
    for b in range(B):
        for (s, e) in sorted(cover[b])[:-1]:
            assert (e - s) % T == 0                      # only a request's last piece is ragged
    if total:
        ideal = -(-(total + (nonempty + d["W"] - 1) * ov) // d["W"])
        assert ideal <= c <= ideal + 2 * PR.MIN_PIECE + PR.CAP_STEP
        assert max(loads) <= c
        cuts = sum(len(cover[b]) - 1 for b in range(B) if lengths[b] > 0)
        assert cuts <= d["W"] - 1 and d["P"] <= 2 * cuts
        for b in range(B):
            if len(cover[b]) > 1:
                assert all(e - s >= PR.MIN_PIECE for (s, e) in cover[b])
    else:
        assert c == 0 and d["n"] == 0
    # workspace holds P partial states
    assert ws >= PR.WS_HEADER_BYTES + d["P"] * H * (512 + 1) * 4 and ws % 256 == 0
    return d


@pytest.mark.parametrize("H", [16, 32, 64, 128])
def test_random_batches(H):
    rng = np.random.default_rng(H)
    for trial in range(20):
        B = int(rng.integers(1, 300))
        L = rng.integers(0, 5000, size=B)
        if trial % 3 == 0:
            L[rng.integers(0, B)] = int(rng.integers(20000, 140000))
        indptr = np.concatenate([[0], np.cumsum(L)]).astype(np.int64)
        _check(indptr, H, int(rng.choice([148, 152, 160, 2, 3])))


def test_edge_batches():
    for H in (16, 128):
        _check([0], H, 152)                       # B = 0
        _check([0, 0, 0], H, 152)                 # only empty requests
        _check([0, 1], H, 152)                    # one token
        _check([0, 131072], H, 152)               # one long request: split across all workers
        _check([0, 65536, 196608], H, 152)
        _check([0, 7, 7, 40, 2000], H, 152)       # empty in the middle


def test_long_request_is_split_over_workers():
    d = _check([0, 65536, 196608], 128, 152)
    assert d["P"] >= d["W"] - 1                     # both requests cut into many pieces
    W = d["W"]
    tokens = [sum(e - s for (_, s, e, _) in d["items"][d["wptr"][w]:d["wptr"][w + 1]]) for w in range(W)]
    perfect = -(-196608 // W)
    assert max(tokens) <= perfect + 2 * PR.ITEM_OVERHEAD[d["variant"]] + PR.MIN_PIECE + PR.CAP_STEP


def test_uniform_batch_cuts_few_requests():
    # 128 requests of 64 tiles on 76 workers: perfect balance needs cuts, but
    # only at worker boundaries
    d = _check([4096 * i for i in range(129)], 128, 152)
    assert d["P"] <= 2 * (d["W"] - 1)
    assert d["n"] <= 128 + d["W"] - 1


def test_unsupported_heads():
    for H in (0, 8, 24, 136, 256):
        with pytest.raises(ValueError):
            PR.build_plan([0, 5], H, 152)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_benchmark_workload_plans(n):
    # the five workloads the bench and the parity tests use, at 152 SMs: every
    # pin above, and the tiles per worker never above the budget's whole tiles
    from mla_latent_kv_absorbed_gb300 import workloads
    b = workloads.make_workload(n)
    d = _check([int(x) for x in b.kv_indptr], b.heads, 152)
    W, T = d["W"], d["T"]
    ov = PR.ITEM_OVERHEAD[d["variant"]]
    for w in range(W):
        its = d["items"][d["wptr"][w]:d["wptr"][w + 1]]
        tiles = sum(-(-(e - s) // T) for (_, s, e, _) in its)
        assert tiles * T + len(its) * ov <= d["c"]
