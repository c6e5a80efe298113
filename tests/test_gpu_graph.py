"""GPU tests of mla_decode_run_graph: one CUDA graph captured once, replayed
after new plans, CSR arrays, queries and cache rows are written into the same
fixed-capacity buffers -- the plan/replay split of "Attention backends",
paragraph "Paged, ragged batches" -- against the fp64 oracle."""
import numpy as np
import pytest

from tests._helpers import assert_close

pytestmark = pytest.mark.gpu

MAX_BATCH = 6
POOL = 8192


def _setup(H):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    words, wsb = binding.decode_graph_sizes(MAX_BATCH, H, sms)
    z = lambda *shape, dt=torch.float32: torch.zeros(shape, dtype=dt, device="cuda")
    buf = dict(plan=z(words, dt=torch.int32), indptr=z(MAX_BATCH + 1, dt=torch.int32), indices=z(16384, dt=torch.int32),
               qn=z(MAX_BATCH, H, 512, dt=torch.bfloat16), qr=z(MAX_BATCH, H, 64, dt=torch.bfloat16),
               kv=z(POOL, 576, dt=torch.bfloat16), out=z(MAX_BATCH, H, 512), lse=z(MAX_BATCH, H),
               ws=z(wsb, dt=torch.uint8))
    return sms, buf


def _load(buf, H, sms, lengths, seed, plan_batch=None):
    """Write a batch into the buffers; the plan covers len(lengths) requests
    (or plan_batch, padding with empty requests); kv_indptr is padded."""
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    bt = W.make_batch(lengths, heads=H, pool=POOL, seed=seed)
    B = len(lengths)
    nb = plan_batch or B
    indptr_plan = np.concatenate([bt.kv_indptr, np.full(nb - B, bt.kv_indptr[-1])]).astype(np.int32)
    plan, _ = binding.decode_plan(indptr_plan, H, sms)
    assert plan.size <= buf["plan"].numel()
    buf["plan"][:plan.size].copy_(torch.from_numpy(plan))
    padded = np.concatenate([bt.kv_indptr, np.full(MAX_BATCH - B, bt.kv_indptr[-1])]).astype(np.int32)
    buf["indptr"].copy_(torch.from_numpy(padded))
    buf["indices"][:bt.nnz].copy_(torch.from_numpy(bt.kv_indices.astype(np.int32)))
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    buf["qn"][:B].copy_(bf(bt.q_nope))
    buf["qr"][:B].copy_(bf(bt.q_rope))
    buf["kv"].copy_(bf(bt.kv_cache))
    buf["out"].fill_(float("nan"))
    buf["lse"].fill_(float("nan"))
    return bt


def _run(buf, H, sms, stream=None):
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    binding.decode_run_graph(buf["plan"], MAX_BATCH, H, sms, buf["qn"], buf["qr"], buf["kv"], buf["indptr"],
                             buf["indices"], W.SM_SCALE, buf["out"], buf["lse"], buf["ws"], stream=stream)


def _check(buf, bt):
    from oracle import mla_oracle as O
    B = bt.batch
    ro, rl = O.decode_attention(bt.q_nope, bt.q_rope, bt.kv_cache, bt.kv_indptr, bt.kv_indices, bt.sm_scale)
    assert_close(buf["out"][:B].cpu().numpy(), buf["lse"][:B].cpu().numpy(), ro, rl)


@pytest.mark.parametrize("H", [16, 128])
def test_one_capture_replayed_with_new_plans(H):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    sms, buf = _setup(H)
    long_len = 3000 if H == 16 else 1500
    cases = [
        ([1, 700, long_len, 64, 0, 129], None),          # full batch, one empty request
        ([2 * long_len, 10, 2], None),                    # fewer requests than the capture (kv_indptr padded)
        ([2 * long_len, 10, 2], MAX_BATCH),               # the same, planned with empty requests up to the capacity
        ([640] * MAX_BATCH, None),                        # equal lengths: a different cut pattern
    ]
    bt = _load(buf, H, sms, cases[0][0], seed=900 + H, plan_batch=cases[0][1])
    _run(buf, H, sms)                                     # eager once, then capture on a side stream
    torch.cuda.synchronize()
    assert binding.check_errors(buf["ws"]) == 0
    _check(buf, bt)
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            _run(buf, H, sms, stream=cap)
    torch.cuda.current_stream().wait_stream(cap)
    for i, (lengths, nb) in enumerate(cases):
        bt = _load(buf, H, sms, lengths, seed=910 + 10 * i + H, plan_batch=nb)
        g.replay()
        torch.cuda.synchronize()
        assert binding.check_errors(buf["ws"]) == 0, (i, lengths)
        _check(buf, bt)


@pytest.mark.parametrize("H", [16, 128])
def test_bad_device_plan_is_reported_not_followed(H):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    sms, buf = _setup(H)
    _load(buf, H, sms, [300, 90], seed=950 + H)
    buf["plan"][0] = 0                                    # wrong magic
    _run(buf, H, sms)
    assert binding.check_errors(buf["ws"]) == 7           # MLA_ERR_PLAN_MISMATCH
    assert torch.isnan(buf["out"][:2]).all()              # nothing computed
    # a plan made for another SM count has another worker count
    bt = _load(buf, H, sms, [300, 90], seed=951 + H)
    plan, _ = binding.decode_plan(bt.kv_indptr, H, sms - 4)
    buf["plan"][:plan.size].copy_(torch.from_numpy(plan))
    _run(buf, H, sms)
    assert binding.check_errors(buf["ws"]) == 7
    # a plan whose item count runs past the buffer's capacity
    bt = _load(buf, H, sms, [300, 90], seed=952 + H)
    buf["plan"][8] = buf["plan"].numel()                  # kHItems
    _run(buf, H, sms)
    assert binding.check_errors(buf["ws"]) == 7
