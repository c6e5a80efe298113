"""GPU parity of the FP8 (E4M3) latent cache path -- mla_decode_run_fp8 and
mla_append_kv_fp8 -- against the fp64 oracle's decode over the dequantised
cache (code value x kv_scale) and its quantiser."""
import numpy as np
import pytest

from tests._helpers import assert_close

pytestmark = pytest.mark.gpu


def _fp8_case(lengths, H, seed, pool=None, q_scale=None):
    from mla_latent_kv_absorbed_gb300 import workloads as W
    pool = pool or max(64, int(sum(lengths)) + 37)
    bt = W.make_batch(lengths, heads=H, pool=pool, seed=seed)   # lengths, slots, q; its bf16 cache is not used
    indices = bt.kv_indices.astype(np.int32)
    codes = W.make_fp8_cache(pool, seed + 2)
    qn, qr = bt.q_nope, bt.q_rope
    if q_scale is not None:                                   # per-head magnitudes far from 1
        f = np.asarray(q_scale, dtype=np.float32)[None, :, None]
        qn = W.f32_to_bf16_bits(_bf16_to_f32(qn) * f)
        qr = W.f32_to_bf16_bits(_bf16_to_f32(qr) * f)
    return bt, qn, qr, codes, indices


def _bf16_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _run_fp8(bt, qn, qr, codes, indices, kv_scale, out_dtype="f32", repeat=1, num_sms=0, kv_dev=None):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    H, B = bt.heads, bt.batch
    plan, _ = binding.decode_plan(bt.kv_indptr, H, num_sms)
    plan_d = torch.from_numpy(plan).cuda()
    ws = torch.zeros(binding.decode_fp8_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    kv = kv_dev if kv_dev is not None else torch.from_numpy(np.ascontiguousarray(codes)).cuda()
    ptr = torch.from_numpy(bt.kv_indptr.astype(np.int32)).cuda()
    idx = torch.from_numpy(indices if indices.size else np.zeros(1, np.int32)).cuda()
    q_n, q_r = bf(qn), bf(qr)
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    res = []
    for _ in range(repeat):
        out = torch.full((B, H, 512), float("nan"), dtype=dt, device="cuda")
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
        binding.decode_run_fp8(plan, plan_d, q_n, q_r, kv, kv_scale, ptr, idx, bt.sm_scale, out, lse, ws)
        st = binding.check_errors(ws)
        assert st == 0, binding.status_string(st)
        res.append((out.float().cpu().numpy(), lse.cpu().numpy()))
    return res if repeat > 1 else res[0]


def _oracle(bt, qn, qr, codes, indices, kv_scale, requests=None):
    from oracle import mla_oracle as O
    return O.decode_attention_fp8(qn, qr, codes, kv_scale, bt.kv_indptr, indices, bt.sm_scale, requests=requests)


@pytest.mark.parametrize("H", [16, 128])
def test_fp8_every_request_empty(H):
    # no plan items: the plan's merge alone writes zeros and lse = -inf
    bt, qn, qr, codes, indices = _fp8_case([0, 0, 0, 0], H, seed=41)
    out, lse = _run_fp8(bt, qn, qr, codes, indices, 2.0 ** -5)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("H", [16, 32, 48, 64, 96, 128])
@pytest.mark.parametrize("lengths", [
    [1, 7, 33, 100],
    [63, 64, 65, 127, 128, 129, 0, 191],          # around the tile edges, an empty request
    [3000, 5, 2100, 640],                          # long requests: cut and merged
])
def test_fp8_decode_matches_oracle(H, lengths):
    from mla_latent_kv_absorbed_gb300 import workloads as W
    bt, qn, qr, codes, idx = _fp8_case(lengths, H, seed=300 + H + len(lengths))
    out, lse = _run_fp8(bt, qn, qr, codes, idx, W.FP8_KV_SCALE)
    ro, rl = _oracle(bt, qn, qr, codes, idx, W.FP8_KV_SCALE)
    assert_close(out, lse, ro, rl)


@pytest.mark.parametrize("H", [16, 32, 128])
def test_fp8_bf16_output_and_many_workers(H):
    from mla_latent_kv_absorbed_gb300 import workloads as W
    rng = np.random.default_rng(H)
    lengths = [int(x) for x in rng.integers(1, 900, size=24)]
    bt, qn, qr, codes, idx = _fp8_case(lengths, H, seed=400 + H)
    out, lse = _run_fp8(bt, qn, qr, codes, idx, W.FP8_KV_SCALE, out_dtype="bf16", num_sms=40)
    ro, rl = _oracle(bt, qn, qr, codes, idx, W.FP8_KV_SCALE)
    assert_close(out, lse, ro, rl)


@pytest.mark.parametrize("H", [16, 128])
def test_fp8_query_heads_of_very_different_magnitude(H):
    # each head is scaled by its own factor: tiny, huge and all-zero heads, the same for the
    # few-heads kernel and the two-CTA kernel (H >= 48), whose exchanged partial scores carry
    # 2^-22 of their half row's largest value whatever its magnitude
    base = [1e-3, 1e3, 0.0, 1.0, 3e-6, 40.0, 1.0, 1.0, 0.02, 1.0, 1.0, 7.0, 1.0, 1.0, 1.0, 250.0]
    bt, qn, qr, codes, idx = _fp8_case([700, 90], H, seed=510 + H, q_scale=(base * (H // 16))[:H])
    for kv_scale in (2.0 ** -5, 0.0123):
        out, lse = _run_fp8(bt, qn, qr, codes, idx, kv_scale)
        ro, rl = _oracle(bt, qn, qr, codes, idx, kv_scale)
        assert_close(out, lse, ro, rl)


@pytest.mark.parametrize("H", [32, 128])
def test_fp8_decode_is_deterministic(H):
    from mla_latent_kv_absorbed_gb300 import workloads as W
    bt, qn, qr, codes, idx = _fp8_case([2500, 300, 1], H, seed=520 + H)
    runs = _run_fp8(bt, qn, qr, codes, idx, W.FP8_KV_SCALE, repeat=3)
    for o, l in runs[1:]:
        assert np.array_equal(o, runs[0][0]) and np.array_equal(l, runs[0][1])


def test_fp8_out_of_range_index_is_reported():
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    bt, qn, qr, codes, idx = _fp8_case([40, 70], 16, seed=530, pool=200)
    idx = idx.copy()
    idx[50] = 200                                  # one past the pool
    plan, _ = binding.decode_plan(bt.kv_indptr, 16)
    ws = torch.zeros(binding.decode_fp8_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    out = torch.empty((2, 16, 512), device="cuda")
    lse = torch.empty((2, 16), device="cuda")
    binding.decode_run_fp8(plan, torch.from_numpy(plan).cuda(), bf(qn), bf(qr), torch.from_numpy(codes).cuda(),
                           W.FP8_KV_SCALE, torch.from_numpy(bt.kv_indptr.astype(np.int32)).cuda(),
                           torch.from_numpy(idx).cuda(), bt.sm_scale, out, lse, ws)
    assert binding.check_errors(ws) == 6           # MLA_ERR_INDEX_OOB


def test_fp8_append_matches_the_oracle_quantiser():
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    from oracle import mla_oracle as O
    rng = np.random.default_rng(540)
    pool, B = 500, 33
    codes = W.make_fp8_cache(pool, 541)
    x = rng.standard_normal((B, 576)).astype(np.float32) * np.exp2(rng.uniform(-12, 12, (B, 1))).astype(np.float32)
    x[0, :8] = [0.0, -0.0, 1e30, -1e30, 448 * 0.0123, 464 * 0.0123, 2.0 ** -20, -(2.0 ** -20)]
    rows = W.f32_to_bf16_bits(x)
    slots = rng.permutation(pool)[:B].astype(np.int32)
    for kv_scale in (W.FP8_KV_SCALE, 0.0123):
        kv = torch.from_numpy(codes.copy()).cuda()
        binding.append_kv_fp8(kv, torch.from_numpy(slots).cuda(),
                              torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).cuda(), kv_scale)
        torch.cuda.synchronize()
        assert np.array_equal(kv.cpu().numpy(), O.append_rows_fp8(codes, slots, rows, kv_scale))


def test_fp8_append_then_decode_step():
    # a decode step over an FP8 cache: quantise the new rows into their slots, then attend
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    from oracle import mla_oracle as O
    lengths = [5, 130, 700]
    bt, qn, qr, codes, idx = _fp8_case(lengths, 16, seed=550)
    new_slots = idx[np.cumsum(lengths) - 1].astype(np.int32)
    rows = W.f32_to_bf16_bits(np.random.default_rng(551).standard_normal((3, 576)).astype(np.float32))
    kv = torch.from_numpy(codes.copy()).cuda()
    binding.append_kv_fp8(kv, torch.from_numpy(new_slots).cuda(),
                          torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).cuda(), W.FP8_KV_SCALE)
    torch.cuda.synchronize()
    after = kv.cpu().numpy()
    assert np.array_equal(after, O.append_rows_fp8(codes, new_slots, rows, W.FP8_KV_SCALE))
    out, lse = _run_fp8(bt, qn, qr, after, idx, W.FP8_KV_SCALE)
    ro, rl = _oracle(bt, qn, qr, after, idx, W.FP8_KV_SCALE)
    assert_close(out, lse, ro, rl)


def test_fp8_full_size_v2lite_sampled():
    # the bench's FP8 leg: V2-Lite-shaped batch (B=64, H=16, contexts U[512, 4096], 2^19-slot pool),
    # every request's lse and a sample of requests' outputs against the oracle
    from mla_latent_kv_absorbed_gb300 import workloads as W
    bt = W.make_workload(2)
    codes = W.make_fp8_cache(bt.pool, 20261200 + 82)
    out, lse = _run_fp8(bt, bt.q_nope, bt.q_rope, codes, bt.kv_indices, W.FP8_KV_SCALE)
    reqs = [0, 1, 17, 40, 63]
    ro, rl = _oracle(bt, bt.q_nope, bt.q_rope, codes, bt.kv_indices, W.FP8_KV_SCALE, requests=reqs)
    assert_close(out, lse, ro, rl, requests=reqs)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_fp8_full_size_v3_sampled():
    # V3-shaped batch (B=128, H=128, 4096 tokens each) over an FP8 cache: the two-CTA kernel,
    # every lse and a sample of requests' outputs against the oracle
    from mla_latent_kv_absorbed_gb300 import workloads as W
    bt = W.make_workload(3)
    codes = W.make_fp8_cache(bt.pool, 20261200 + 83)
    out, lse = _run_fp8(bt, bt.q_nope, bt.q_rope, codes, bt.kv_indices, W.FP8_KV_SCALE)
    reqs = [0, 63, 127]
    ro, rl = _oracle(bt, bt.q_nope, bt.q_rope, codes, bt.kv_indices, W.FP8_KV_SCALE, requests=reqs)
    assert_close(out, lse, ro, rl, requests=reqs)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("H", [16, 128])
def test_fp8_rows_past_4_gib_of_the_pool(H):
    # every row the batch reads sits above slot 2^23 of a 4.8 GB FP8 pool (byte
    # offsets past 2^32); the result equals the oracle on the compact pool
    import torch
    from mla_latent_kv_absorbed_gb300 import workloads as W
    bt, qn, qr, codes, idx = _fp8_case([300, 5, 1000, 64], H, seed=610 + H)
    base, big = 1 << 23, (1 << 23) + 4096
    used = np.unique(idx)
    assert used.size < big - base
    mapping = np.full(codes.shape[0], -1, dtype=np.int64)
    mapping[used] = base + np.arange(used.size)
    pool = torch.zeros((big, 576), dtype=torch.uint8, device="cuda")
    pool[torch.from_numpy(mapping[used]).cuda()] = torch.from_numpy(np.ascontiguousarray(codes[used])).cuda()
    out, lse = _run_fp8(bt, qn, qr, codes, mapping[idx].astype(np.int32), W.FP8_KV_SCALE, kv_dev=pool)
    ro, rl = _oracle(bt, qn, qr, codes, idx, W.FP8_KV_SCALE)
    assert_close(out, lse, ro, rl)
