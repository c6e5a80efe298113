"""GPU parity of the multi-query (draft verification) decode against the fp64
oracle: q_len draft tokens per request, query i causally limited, the q_len x H
query rows read as the heads of one request."""
import numpy as np
import pytest

from tests._helpers import ATOL_LSE, ATOL_OUT, RTOL_OUT

pytestmark = pytest.mark.gpu


def _run(bt, q_len, H, out_dtype="f32", num_sms=0):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    from tests._helpers import to_device
    dev = to_device(bt)
    B = bt.batch
    plan, ws_bytes = binding.decode_plan(bt.kv_indptr, q_len * H, num_sms)
    plan_d = torch.from_numpy(plan).cuda()
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    out = torch.full((B, q_len, H, 512), float("nan"), dtype=dt, device="cuda")
    lse = torch.full((B, q_len, H), float("nan"), dtype=torch.float32, device="cuda")
    binding.decode_run_multi_query(plan, plan_d, q_len, dev["q_nope"], dev["q_rope"], dev["kv_cache"],
                                   dev["kv_indptr"], dev["kv_indices"], bt.sm_scale, out, lse, ws)
    assert binding.check_errors(ws) == 0
    return out.float().cpu().numpy(), lse.cpu().numpy(), plan


def _batch(lengths, q_len, H, seed):
    # a batch whose q arrays hold q_len x H rows per request
    from mla_latent_kv_absorbed_gb300 import workloads as W
    return W.make_batch(lengths, heads=q_len * H, pool=max(64, int(np.sum(lengths)) + 17), seed=seed)


def _check(out, lse, ro, rl):
    err = np.abs(out - ro)
    assert np.isfinite(out).all()
    assert (err <= ATOL_OUT + RTOL_OUT * np.abs(ro)).all(), f"out: max err {err.max():.3e}"
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(lse), fin)
    if fin.any():
        assert np.abs(lse[fin] - rl[fin]).max() <= ATOL_LSE


@pytest.mark.parametrize("q_len,H", [(4, 16), (2, 32), (3, 32), (2, 64), (8, 16), (1, 64),
                                     (2, 8), (4, 4), (2, 16), (4, 8), (16, 2)])   # 16 / 32 rows: few-heads kernel
def test_multi_query_matches_oracle(q_len, H):
    from oracle import mla_oracle as O
    lengths = [q_len, 70, 300, 1500]
    bt = _batch(lengths, q_len, H, seed=90 + 7 * q_len + H)
    out, lse, _ = _run(bt, q_len, H)
    B = bt.batch
    qn = bt.q_nope.reshape(B, q_len, H, 512)
    qr = bt.q_rope.reshape(B, q_len, H, 64)
    ro, rl = O.decode_attention_multi_query(qn, qr, bt.kv_cache, bt.kv_indptr, bt.kv_indices, bt.sm_scale, q_len)
    _check(out, lse, ro, rl)


def test_multi_query_across_cut_requests_and_bf16_output():
    # few workers force cuts inside long requests, so some pieces end inside
    # the drafts and the merge combines causally limited partial states
    from oracle import mla_oracle as O
    q_len, H = 4, 16
    bt = _batch([2500, 1900, 4], q_len, H, seed=123)
    out, lse, plan = _run(bt, q_len, H, out_dtype="bf16", num_sms=6)
    assert plan[10] > 0, "the plan should cut requests"
    B = bt.batch
    ro, rl = O.decode_attention_multi_query(bt.q_nope.reshape(B, q_len, H, 512), bt.q_rope.reshape(B, q_len, H, 64),
                                            bt.kv_cache, bt.kv_indptr, bt.kv_indices, bt.sm_scale, q_len)
    _check(out, lse, ro, rl)


def test_multi_query_short_context_rows_on_both_kernels():
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    q_len, H = 4, 16
    bt = _batch([2, 9], q_len, H, seed=5)            # request 0 holds fewer rows than drafts
    out, lse, _ = _run(bt, q_len, H)
    assert np.all(out[0, :2] == 0) and np.all(np.isneginf(lse[0, :2]))
    assert np.isfinite(lse[0, 2:]).all() and np.isfinite(lse[1]).all()
    # the same on the few-heads kernel (q_len x H = 16 rows)
    from oracle import mla_oracle as O
    bt2 = _batch([2, 9, 130], 4, 4, seed=6)
    out2, lse2, _ = _run(bt2, 4, 4)
    assert np.all(out2[0, :2] == 0) and np.all(np.isneginf(lse2[0, :2]))
    # requests 1 and 2 (at least q_len rows: the oracle's domain) against the oracle
    B = bt2.batch
    ro, rl = O.decode_attention_multi_query(bt2.q_nope.reshape(B, 4, 4, 512)[1:], bt2.q_rope.reshape(B, 4, 4, 64)[1:],
                                            bt2.kv_cache, bt2.kv_indptr[1:], bt2.kv_indices, bt2.sm_scale, 4)
    _check(out2[1:], lse2[1:], ro, rl)
    # a q_len that does not divide the plan's rows is refused
    with pytest.raises(binding.MLAError):
        _run(bt2, 3, 4)


@pytest.mark.slow
@pytest.mark.parametrize("q_len,H", [(4, 16), (2, 16)])
def test_multi_query_full_size_v2lite_sampled(q_len, H):
    # the bench's draft-verification shapes at the V2-Lite contexts (64
    # requests, 512..4096 rows): 64 rows on the two-CTA kernel, 32 on the
    # few-heads kernel, the plan of the whole batch; a sample of requests
    # (as their own CSR batch) against the oracle
    from mla_latent_kv_absorbed_gb300 import workloads as W
    from oracle import mla_oracle as O
    ref = W.make_workload(2)
    bt = W.make_batch([int(x) for x in ref.lengths], heads=q_len * H, pool=ref.pool, seed=1800 + q_len)
    out, lse, _ = _run(bt, q_len, H)
    req = sorted(set([0, bt.batch - 1] + list(range(0, bt.batch, 9))))
    lens = [int(bt.kv_indptr[b + 1] - bt.kv_indptr[b]) for b in req]
    ptr = np.concatenate([[0], np.cumsum(lens)])
    ind = np.concatenate([bt.kv_indices[bt.kv_indptr[b]:bt.kv_indptr[b + 1]] for b in req])
    qn = bt.q_nope[req].reshape(len(req), q_len, H, 512)
    qr = bt.q_rope[req].reshape(len(req), q_len, H, 64)
    ro, rl = O.decode_attention_multi_query(qn, qr, bt.kv_cache, ptr, ind, bt.sm_scale, q_len)
    _check(out[req], lse[req], ro, rl)
