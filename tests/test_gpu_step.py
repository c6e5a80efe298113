"""GPU tests of the cache append (mla_append_kv) and of a whole absorbing decode
step -- absorb, append, decode, project -- run eagerly and captured in a CUDA
graph, against the fp64 oracle."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _bf(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _bits(t):
    import torch
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def test_append_is_exact_and_touches_nothing_else():
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    from oracle import mla_oracle as O
    rng = np.random.default_rng(5)
    pool, B = 3000, 37
    kv = W.f32_to_bf16_bits(rng.standard_normal((pool, 576), dtype=np.float32))
    rows = W.f32_to_bf16_bits(rng.standard_normal((B, 576), dtype=np.float32))
    slots = rng.permutation(pool)[:B].astype(np.int32)
    kv_d = _bf(kv)
    binding.append_kv(kv_d, torch.from_numpy(slots).cuda(), _bf(rows))
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kv_d), O.append_rows(kv, slots, rows))


def test_append_out_of_range_slot_is_reported_and_skipped():
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    rng = np.random.default_rng(6)
    pool = 64
    kv = W.f32_to_bf16_bits(rng.standard_normal((pool, 576), dtype=np.float32))
    rows = W.f32_to_bf16_bits(rng.standard_normal((3, 576), dtype=np.float32))
    slots = np.array([5, pool, -1], dtype=np.int32)
    kv_d = _bf(kv)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    binding.append_kv(kv_d, torch.from_numpy(slots).cuda(), _bf(rows), workspace=ws)
    assert binding.check_errors(ws) == 6               # MLA_ERR_INDEX_OOB
    want = kv.copy()
    want[5] = rows[0]
    assert np.array_equal(_bits(kv_d), want)


@pytest.mark.parametrize("H", [16, 128])
def test_absorbing_step_eager_and_in_a_cuda_graph(H):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    from oracle import mla_oracle as O
    # each request's last token is this step's new row, appended into a free slot
    lengths = [3, 90, 260]
    B = len(lengths)
    bt = W.make_batch(lengths, heads=H, pool=1024, seed=61 + H)
    new_slots = bt.kv_indices[np.cumsum(lengths) - 1].astype(np.int32)
    dec = binding.Decoder(bt.kv_indptr, H)
    kv = _bf(bt.kv_cache)
    indptr = torch.from_numpy(bt.kv_indptr.astype(np.int32)).cuda()
    indices = torch.from_numpy(bt.kv_indices.astype(np.int32)).cuda()
    slots = torch.from_numpy(new_slots).cuda()
    # device buffers the step reads and writes (fixed addresses for the graph)
    q_pre = torch.empty((B, H, 128), dtype=torch.bfloat16, device="cuda")
    q_rope = torch.empty((B, H, 64), dtype=torch.bfloat16, device="cuda")
    rows = torch.empty((B, 576), dtype=torch.bfloat16, device="cuda")
    w_kc = torch.empty((H, 128, 512), dtype=torch.bfloat16, device="cuda")
    w_vc = torch.empty((H, 512, 128), dtype=torch.bfloat16, device="cuda")
    q_lat = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    o_lat = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    out = torch.empty((B, H, 128), dtype=torch.float32, device="cuda")

    def step(stream=None):
        binding.absorb_query(q_pre, w_kc, q_lat, stream=stream)
        binding.append_kv(kv, slots, rows, stream=stream)
        dec.run(q_lat, q_rope, kv, indptr, indices, bt.sm_scale, o_lat, lse, stream=stream)
        binding.project_output(o_lat, w_vc, out, stream=stream)

    def load_inputs(seed):
        x = W.make_head_product_inputs(B, H, seed=seed)
        rng = np.random.default_rng(seed + 1)
        qr = W.f32_to_bf16_bits(rng.standard_normal((B, H, 64), dtype=np.float32))
        nr = W.f32_to_bf16_bits(rng.standard_normal((B, 576), dtype=np.float32))
        for dst, src in ((q_pre, x.q_pre), (w_kc, x.w_kc), (w_vc, x.w_vc), (q_rope, qr), (rows, nr)):
            dst.copy_(_bf(src))
        return x, qr, nr

    def expected(x, qr, nr, q_bits, o_bits):
        cache = O.append_rows(bt.kv_cache, new_slots, nr)
        ro, rl = O.decode_attention(q_bits, qr, cache, bt.kv_indptr, bt.kv_indices, bt.sm_scale)
        return O.absorb_query(O.bf16_bits_to_f64(x.q_pre), O.bf16_bits_to_f64(x.w_kc)), ro, rl, \
            O.project_output(O.bf16_bits_to_f64(o_bits), O.bf16_bits_to_f64(x.w_vc)), cache

    def check(x, qr, nr):
        q_bits, o_bits = _bits(q_lat), _bits(o_lat)
        rq, ro, rl, rp, cache = expected(x, qr, nr, q_bits, o_bits)
        e = lambda a, r, at, rt: np.all(np.abs(a - r) <= at + rt * np.abs(r))
        assert e(O.bf16_bits_to_f64(q_bits), rq, 2e-3, 4e-3), "absorb"
        assert np.array_equal(_bits(kv), cache), "append"
        assert e(O.bf16_bits_to_f64(o_bits), ro, 1e-2, 1e-2), "decode out"
        assert np.max(np.abs(lse.cpu().numpy() - rl)) <= 2e-3, "decode lse"
        assert e(out.cpu().numpy(), rp, 1e-4, 1e-4), "project"

    inp = load_inputs(500)
    step()
    assert dec.check() == 0
    check(*inp)
    eager = out.cpu().numpy().copy()

    # capture once, then replay with new inputs written into the same buffers
    kv.copy_(_bf(bt.kv_cache))
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            step(stream=cap)
    torch.cuda.current_stream().wait_stream(cap)
    kv.copy_(_bf(bt.kv_cache))
    load_inputs(500)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), eager), "replay of the same inputs differs from the eager step"
    kv.copy_(_bf(bt.kv_cache))
    inp2 = load_inputs(777)
    g.replay()
    torch.cuda.synchronize()
    assert dec.check() == 0
    check(*inp2)


@pytest.mark.parametrize("H,out_dtype,pinned_out", [(16, "f32", True), (128, "bf16", True), (128, "f32", True),
                                                    (16, "f32", False), (128, "bf16", False)])
def test_host_buffer_step_equals_device_run(H, out_dtype, pinned_out):
    # the result copied back into page-locked or pageable host buffers: the
    # device run's bits either way
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    from tests._helpers import to_device
    bt = W.make_batch([5, 300, 1, 2100], heads=H, pool=4096, seed=71 + H)
    dev = to_device(bt)
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    dec = binding.Decoder(bt.kv_indptr, H)
    ref_out = torch.empty((bt.batch, H, 512), dtype=dt, device="cuda")
    ref_lse = torch.empty((bt.batch, H), dtype=torch.float32, device="cuda")
    dec.run(dev["q_nope"], dev["q_rope"], dev["kv_cache"], dev["kv_indptr"], dev["kv_indices"], bt.sm_scale,
            ref_out, ref_lse)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hq = pin(bt.q_nope.view(np.int16)).view(torch.bfloat16)
    hr = pin(bt.q_rope.view(np.int16)).view(torch.bfloat16)
    hp, hi = pin(bt.kv_indptr.astype(np.int32)), pin(bt.kv_indices.astype(np.int32))
    out = torch.empty((bt.batch, H, 512), dtype=dt)
    lse = torch.empty((bt.batch, H), dtype=torch.float32)
    if pinned_out:
        out, lse = out.pin_memory(), lse.pin_memory()
    plan = torch.empty(dec.plan_host.shape[0], dtype=torch.int32).pin_memory()
    staging = torch.empty(binding.step_staging_bytes(bt.batch, H, bt.nnz, plan.numel(), 0 if dt == torch.float32 else 1),
                          dtype=torch.uint8, device="cuda")
    ws = torch.zeros(max(dec.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    binding.decode_step_host(hq, hr, hp, hi, dev["kv_cache"], bt.sm_scale, out, lse, plan, staging, ws)
    torch.cuda.synchronize()
    assert binding.check_errors(ws) == 0
    assert np.array_equal(plan.numpy(), dec.plan_host)
    assert torch.equal(out, ref_out.cpu()) and torch.equal(lse, ref_lse.cpu())
