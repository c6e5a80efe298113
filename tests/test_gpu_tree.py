"""GPU parity of tree-shaped draft verification (mla_decode_run_tree) against
the fp64 oracle's decode_attention_tree ("[sglang] EAGLE 트리 검증 어텐션
최적화", section "들어가며": each draft query sees the verified context and
its own ancestor chain among the drafts).

Both decode kernels are covered: W x H rows of 16 or 32 run on the few-heads
kernel, 64 or 128 on the two-CTA kernel.  Requests are also cut across many
workers (a small SM count for the plan) so that pieces begin and end inside
the draft tokens; contexts of exactly W rows have no shared part at all.
"""
import numpy as np
import pytest

from tests._helpers import assert_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_latent_kv_absorbed_gb300 import build
    build.build()


def _random_tree(rng, W):
    return np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, W)], dtype=np.int32)


def _topk_tree(W, k=2):
    # breadth-first expansion: every node gets k children until W nodes exist
    par = [-1]
    i = 0
    while len(par) < W:
        for _ in range(k):
            if len(par) < W:
                par.append(i)
        i += 1
    return np.array(par, dtype=np.int32)


def _run(bt, W, parents, num_sms=0, out_dtype="f32", expect_status=0):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    B, rows = bt.batch, bt.heads
    Hq = rows // W
    dev = to_device(bt)
    plan, ws_bytes = binding.decode_plan(bt.kv_indptr, rows, num_sms)
    plan_d = torch.from_numpy(plan).cuda()
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    par = torch.from_numpy(np.ascontiguousarray(parents, dtype=np.int32)).cuda()
    masks = torch.zeros((B, W), dtype=torch.int64, device="cuda")
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    out = torch.full((B, W, Hq, 512), float("nan"), dtype=dt, device="cuda")
    lse = torch.full((B, W, Hq), float("nan"), dtype=torch.float32, device="cuda")
    binding.decode_run_tree(plan, plan_d, par, masks, dev["q_nope"], dev["q_rope"], dev["kv_cache"],
                            dev["kv_indptr"], dev["kv_indices"], bt.sm_scale, out, lse, ws)
    st = binding.check_errors(ws)
    assert st == expect_status, binding.status_string(st)
    return out.float().cpu().numpy(), lse.cpu().numpy(), masks.cpu().numpy()


def _case(lengths, W, Hq, seed):
    from mla_latent_kv_absorbed_gb300 import workloads as Wl
    return Wl.make_batch(lengths, heads=W * Hq, pool=int(np.sum(lengths)) + 97, seed=seed)


def _oracle(bt, W, parents):
    from oracle import mla_oracle as O
    B, Hq = bt.batch, bt.heads // W
    return O.decode_attention_tree(bt.q_nope.reshape(B, W, Hq, 512), bt.q_rope.reshape(B, W, Hq, 64),
                                   bt.kv_cache, bt.kv_indptr, bt.kv_indices, bt.sm_scale, parents)


@pytest.mark.parametrize("W,Hq", [(4, 4), (8, 4), (2, 16), (4, 16), (8, 16), (64, 2)])
@pytest.mark.parametrize("shape", ["random", "topk2", "star"])
def test_tree_matches_oracle(W, Hq, shape):
    rng = np.random.default_rng(1000 + 10 * W + Hq)
    lengths = [W, W + 1, 700, 64 + W, 3 * 64 + 5, 2000]
    bt = _case(lengths, W, Hq, seed=1100 + W + Hq)
    if shape == "random":
        parents = np.stack([_random_tree(rng, W) for _ in lengths])
    elif shape == "topk2":
        parents = np.tile(_topk_tree(W), (len(lengths), 1))
    else:
        parents = np.full((len(lengths), W), -1, dtype=np.int32)
    out, lse, masks = _run(bt, W, parents)
    ro, rl = _oracle(bt, W, parents)
    assert_close(out.reshape(bt.batch, -1, 512), lse.reshape(bt.batch, -1), ro.reshape(bt.batch, -1, 512),
                 rl.reshape(bt.batch, -1))
    # the mask words are the ancestor-or-self sets
    from oracle import mla_oracle as O
    for b in range(len(lengths)):
        for i, anc in enumerate(O.tree_ancestors(parents[b])):
            assert (int(masks[b, i]) & ((1 << 64) - 1)) == sum(1 << a for a in anc)


@pytest.mark.parametrize("W,Hq,num_sms", [(8, 4, 9), (8, 16, 7), (4, 16, 40), (64, 2, 5)])
def test_tree_on_requests_cut_across_workers(W, Hq, num_sms):
    # long contexts cut into many pieces: pieces that start and end inside the
    # drafts, merged by LSE afterwards
    rng = np.random.default_rng(1200 + W + num_sms)
    lengths = [9000 + 37, 4100, 64 * 7 + 3, 12000 + 61]
    bt = _case(lengths, W, Hq, seed=1300 + W + num_sms)
    parents = np.stack([_random_tree(rng, W) for _ in lengths])
    out, lse, _ = _run(bt, W, parents, num_sms=num_sms)
    ro, rl = _oracle(bt, W, parents)
    assert_close(out.reshape(bt.batch, -1, 512), lse.reshape(bt.batch, -1), ro.reshape(bt.batch, -1, 512),
                 rl.reshape(bt.batch, -1))


@pytest.mark.parametrize("W,Hq", [(4, 4), (8, 16)])
def test_chain_tree_equals_the_multi_query_path(W, Hq):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    lengths = [W + 3, 900, 4000]
    bt = _case(lengths, W, Hq, seed=1400 + W)
    chain = np.tile(np.arange(-1, W - 1, dtype=np.int32), (len(lengths), 1))
    out, lse, _ = _run(bt, W, chain)
    dev = to_device(bt)
    plan, ws_bytes = binding.decode_plan(bt.kv_indptr, W * Hq)
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    o2 = torch.empty((bt.batch, W, Hq, 512), device="cuda")
    l2 = torch.empty((bt.batch, W, Hq), device="cuda")
    binding.decode_run_multi_query(plan, torch.from_numpy(plan).cuda(), W, dev["q_nope"], dev["q_rope"],
                                   dev["kv_cache"], dev["kv_indptr"], dev["kv_indices"], bt.sm_scale, o2, l2, ws)
    assert binding.check_errors(ws) == 0
    assert_close(out, lse, o2.cpu().numpy(), l2.cpu().numpy())
    ro, rl = _oracle(bt, W, chain)
    assert_close(out.reshape(bt.batch, -1, 512), lse.reshape(bt.batch, -1), ro.reshape(bt.batch, -1, 512),
                 rl.reshape(bt.batch, -1))


def test_tree_bf16_output():
    rng = np.random.default_rng(1500)
    W, Hq = 8, 16
    lengths = [300, 2500, 8]
    bt = _case(lengths, W, Hq, seed=1500)
    parents = np.stack([_random_tree(rng, W) for _ in lengths])
    out, lse, _ = _run(bt, W, parents, out_dtype="bf16")
    ro, rl = _oracle(bt, W, parents)
    assert_close(out.reshape(bt.batch, -1, 512), lse.reshape(bt.batch, -1), ro.reshape(bt.batch, -1, 512),
                 rl.reshape(bt.batch, -1))


@pytest.mark.parametrize("W,Hq", [(4, 4), (4, 16)])
def test_bad_parent_is_reported_and_verified_as_a_child_of_the_context(W, Hq):
    lengths = [500, 40]
    bt = _case(lengths, W, Hq, seed=1600 + Hq)
    parents = np.tile(_topk_tree(W), (2, 1))
    bad = parents.copy()
    bad[1, 2] = 3                                  # not an earlier draft
    out, lse, masks = _run(bt, W, bad, expect_status=8)     # MLA_ERR_TREE
    assert int(masks[1, 2]) == 1 << 2
    fixed = parents.copy()
    fixed[1, 2] = -1
    ro, rl = _oracle(bt, W, fixed)
    assert_close(out.reshape(bt.batch, -1, 512), lse.reshape(bt.batch, -1), ro.reshape(bt.batch, -1, 512),
                 rl.reshape(bt.batch, -1))


def _sub_batch(bt, W, requests):
    """The given requests of a batch as their own CSR batch (their rows, their
    queries), for the oracle."""
    import copy
    sub = copy.copy(bt)
    lens = [int(bt.kv_indptr[b + 1] - bt.kv_indptr[b]) for b in requests]
    sub.kv_indptr = np.concatenate([[0], np.cumsum(lens)]).astype(bt.kv_indptr.dtype)
    sub.kv_indices = np.concatenate([bt.kv_indices[bt.kv_indptr[b]:bt.kv_indptr[b + 1]] for b in requests])
    sub.q_nope, sub.q_rope = bt.q_nope[requests], bt.q_rope[requests]
    sub.lengths = np.asarray(lens, dtype=bt.lengths.dtype)
    return sub


@pytest.mark.slow
@pytest.mark.parametrize("shape", ["topk2", "chain"])
def test_tree_full_size_v2lite_sampled(shape):
    # the bench's draft-verification shape: the V2-Lite contexts (64 requests,
    # 512..4096 rows), 8 drafts of 16 heads (128 rows, the two-CTA kernel),
    # the plan of the whole batch; a sample of requests against the oracle
    from mla_latent_kv_absorbed_gb300 import workloads as Wl
    W, Hq = 8, 16
    ref = Wl.make_workload(2)
    bt = Wl.make_batch([int(x) for x in ref.lengths], heads=W * Hq, pool=ref.pool, seed=1700)
    parents = np.tile(_topk_tree(W) if shape == "topk2" else np.arange(-1, W - 1, dtype=np.int32),
                      (bt.batch, 1)).astype(np.int32)
    out, lse, _ = _run(bt, W, parents)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    req = sorted(set([0, bt.batch - 1] + list(range(0, bt.batch, 9))))
    sub = _sub_batch(bt, W, req)
    ro, rl = _oracle(sub, W, parents[req])
    assert_close(out[req].reshape(len(req), -1, 512), lse[req].reshape(len(req), -1),
                 ro.reshape(len(req), -1, 512), rl.reshape(len(req), -1))
