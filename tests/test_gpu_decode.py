"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, on
seeded synthetic batches.  Bar: |dout| <= 1e-2 + 1e-2|ref|, |dlse| <= 2e-3;
identical results on repeated runs and under slot relabelling."""
import numpy as np
import pytest

from tests._helpers import assert_close, oracle, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_latent_kv_absorbed_gb300 import build
    build.build()


def _batch(lengths, heads, pool=None, seed=0, slots="permutation"):
    from mla_latent_kv_absorbed_gb300 import workloads as W
    nnz = int(np.sum(lengths))
    pool = pool or max(64, nnz + 17)
    return W.make_batch(lengths, heads=heads, pool=pool, seed=seed, slots=slots)


def test_tiny_workload_full():
    from mla_latent_kv_absorbed_gb300 import workloads as W
    bt = W.make_workload(1)
    (out, lse), dec = run_gpu(bt)
    ro, rl = oracle(bt)
    assert_close(out, lse, ro, rl)
    assert dec.header[4] == 1   # few-heads kernel variant ran


@pytest.mark.parametrize("H", [16, 32, 48, 64, 80, 96, 112, 128])
def test_ragged_tails_small(H):
    # lengths around the 128-token tile edges, plus an empty request
    bt = _batch([1, 2, 3, 127, 128, 129, 0, 255, 256, 257, 1000, 64], H, seed=H)
    (out, lse), _ = run_gpu(bt)
    ro, rl = oracle(bt)
    assert_close(out, lse, ro, rl)


@pytest.mark.parametrize("H", [16, 32, 128])
def test_split_and_merge_long_request(H):
    # one long request is cut over every worker and merged by LSE
    bt = _batch([20000, 3], H, seed=7)
    (out, lse), dec = run_gpu(bt)
    assert dec.header[9] > 1   # partial states were used
    ro, rl = oracle(bt)
    assert_close(out, lse, ro, rl)


@pytest.mark.parametrize("H", [16, 128])
def test_bf16_output(H):
    import torch
    bt = _batch([100, 513, 1], H, seed=3)
    (out, lse), _ = run_gpu(bt, out_dtype=torch.bfloat16)
    ro, rl = oracle(bt)
    assert_close(out, lse, ro, rl)


def test_lse_optional_and_duplicate_slots():
    from mla_latent_kv_absorbed_gb300 import workloads as W
    bt = _batch([50, 70], 16, seed=4)
    bt.kv_indices[10:20] = bt.kv_indices[0:10]    # a slot named twice counts twice
    (out, lse), _ = run_gpu(bt, with_lse=False)
    ro, rl = oracle(bt)
    assert lse is None
    assert_close(out, None, ro, rl)


@pytest.mark.parametrize("H", [16, 128])
def test_repeat_runs_bit_identical_and_slot_relabelling(H):
    bt = _batch([300, 1, 4000, 77], H, seed=5)
    runs, _ = run_gpu(bt, repeat=2)
    (o1, l1), (o2, l2) = runs
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    perm = np.random.default_rng(1).permutation(bt.pool)
    kv2 = np.empty_like(bt.kv_cache)
    kv2[perm] = bt.kv_cache
    bt.kv_cache = kv2
    bt.kv_indices = perm[bt.kv_indices].astype(np.int32)
    (o3, l3), _ = run_gpu(bt)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)


@pytest.mark.parametrize("H", [16, 128])
def test_forced_chunkings_agree(H):
    # different SM counts give different plans; all must match the oracle
    bt = _batch([3000, 5000, 12, 900], H, seed=6)
    ro, rl = oracle(bt)
    dev = to_device(bt)
    for sms in ((152, 40, 7, 1) if H <= 32 else (152, 40, 8, 2)):
        (out, lse), dec = run_gpu(bt, dev=dev, num_sms=sms)
        assert_close(out, lse, ro, rl)


def test_index_out_of_range_is_reported_not_faulted():
    from mla_latent_kv_absorbed_gb300 import binding
    import torch
    bt = _batch([40, 40], 16, seed=8)
    bt.kv_indices[5] = bt.pool + 100
    dev = to_device(bt)
    dec = binding.Decoder(bt.kv_indptr, 16)
    out = torch.empty((2, 16, 512), device="cuda")
    dec.run(dev["q_nope"], dev["q_rope"], dev["kv_cache"], dev["kv_indptr"], dev["kv_indices"],
            bt.sm_scale, out, None)
    assert dec.check() == 6          # MLA_ERR_INDEX_OOB
    assert dec.check() == 0          # status cleared


@pytest.mark.slow
def test_v2lite_workload_sampled():
    from mla_latent_kv_absorbed_gb300 import workloads as W
    bt = W.make_workload(2)
    (out, lse), _ = run_gpu(bt)
    req = list(range(0, bt.batch, 7))
    ro, rl = oracle(bt, requests=req)
    assert_close(out, lse, ro, rl, requests=req)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("H", [16, 128])
def test_attend_then_merge_equals_run(H):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    bt = _batch([9000, 40, 3000], H, seed=12)
    dev = to_device(bt)
    dec = binding.Decoder(bt.kv_indptr, H)
    assert dec.has_merge
    outs = []
    for mode in ("run", "split"):
        out = torch.full((bt.batch, H, 512), float("nan"), device="cuda")
        lse = torch.full((bt.batch, H), float("nan"), device="cuda")
        args = (dev["q_nope"], dev["q_rope"], dev["kv_cache"], dev["kv_indptr"], dev["kv_indices"], bt.sm_scale,
                out, lse)
        if mode == "run":
            dec.run(*args)
        else:
            dec.attend(*args)
            dec.merge(out, lse)
        assert dec.check() == 0
        outs.append((out.cpu().numpy(), lse.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("H,counts", [(16, [3, 1, 0, 5]), (5, [2, 40, 0, 1, 70, 33]), (24, [9, 17, 4])])
def test_public_merge_states_matches_oracle_merge(H, counts):
    # head counts that are not a multiple of a block's heads; more than 32
    # partials for one warp (the LSEs are taken 32 at a time)
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    from oracle import mla_oracle as O
    rng = np.random.default_rng(3 + H)
    P = sum(counts)
    vp = rng.standard_normal((P, H, 512)).astype(np.float32)
    sp = (rng.standard_normal((P, H)) * 4).astype(np.float32)
    sp[1, :3] = -np.inf                       # empty partials carry no weight
    if counts[-1] > 32:
        sp[-1, :] += 30.0                     # the last chunk raises the running maximum
    ind = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    out = torch.empty((len(counts), H, 512), device="cuda")
    lse = torch.empty((len(counts), H), device="cuda")
    binding.merge_states(torch.from_numpy(vp).cuda(), torch.from_numpy(sp).cuda(), torch.from_numpy(ind).cuda(),
                         out, lse)
    torch.cuda.synchronize()
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(len(counts)):
        ro, rl = O.merge_states(vp[ind[b]:ind[b + 1]].astype(np.float64), sp[ind[b]:ind[b + 1]].astype(np.float64))
        np.testing.assert_allclose(o[b], ro, rtol=1e-5, atol=1e-5)
        fin = np.isfinite(rl)
        np.testing.assert_allclose(l[b][fin], rl[fin], atol=1e-5)
        assert np.all(np.isneginf(l[b][~fin]))


def test_pair_kernel_variant_and_empty_requests():
    bt = _batch([0, 65, 0, 200, 0], 128, seed=13)
    (out, lse), dec = run_gpu(bt)
    assert dec.header[4] == 2   # two-CTA cluster variant ran
    ro, rl = oracle(bt)
    assert_close(out, lse, ro, rl)
    assert np.all(out[[0, 2, 4]] == 0)


@pytest.mark.parametrize("H", [16, 128])
def test_every_request_empty(H):
    # a plan without items: nothing is gathered, and the plan's merge alone
    # writes a zero output and lse = -inf for every request
    import torch
    bt = _batch([0, 0, 0], H, seed=5)
    for dt in (torch.float32, torch.bfloat16):
        (out, lse), dec = run_gpu(bt, out_dtype=dt)
        assert dec.header[8] == 0 and dec.header[10] == 3
        assert np.all(out == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("H", [16, 128])
def test_empty_batch_is_a_no_op(H):
    bt = _batch([], H, seed=6)
    (out, lse), dec = run_gpu(bt)
    assert dec.header[2] == 0 and out.shape == (0, H, 512) and lse.shape == (0, H)


@pytest.mark.slow
@pytest.mark.parametrize("number", [3, 4, 5])
def test_many_head_workloads_sampled(number):
    from mla_latent_kv_absorbed_gb300 import workloads as W
    bt = W.make_workload(number)
    (out, lse), _ = run_gpu(bt)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    req = sorted(set([0, bt.batch - 1] + list(range(0, bt.batch, max(1, bt.batch // 6)))))
    ro, rl = oracle(bt, requests=req)
    assert_close(out, lse, ro, rl, requests=req)


@pytest.mark.parametrize("H", [16, 128])
def test_plan_item_outside_its_request_is_reported_not_faulted(H):
    # A plan item naming the wrong request (its tokens still inside kv_indices)
    # and one reaching past kv_indices: the call returns, the device status
    # reads MLA_ERR_PLAN_MISMATCH, and the next call with a good plan is clean.
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    bt = _batch([300, 200, 500], H, seed=21)
    dev = to_device(bt)
    dec = binding.Decoder(bt.kv_indptr, H)
    W = int(dec.plan_host[6])
    items_off = 16 + W + 1
    bad = dec.plan_host.copy()
    bad[items_off] = (bad[items_off] + 1) % bt.batch          # first item now names another request
    n_items = int(bad[8])
    bad[items_off + 4 * (n_items - 1) + 2] = bt.nnz + 64      # last item reaches past kv_indices
    out = torch.zeros((bt.batch, H, 512), device="cuda")
    lse = torch.zeros((bt.batch, H), device="cuda")
    # straight through the C ABI: the binding would refuse this plan on the
    # host (its last item reaches past kv_indices); the kernels must cope too
    import ctypes
    bad_d = torch.from_numpy(bad).cuda()
    st = binding.library().mla_decode_run(
        bad.ctypes.data, bad_d.data_ptr(), dev["q_nope"].data_ptr(), dev["q_rope"].data_ptr(),
        dev["kv_cache"].data_ptr(), bt.pool, dev["kv_indptr"].data_ptr(), dev["kv_indices"].data_ptr(),
        ctypes.c_float(bt.sm_scale), out.data_ptr(), 0, lse.data_ptr(), dec.workspace.data_ptr(),
        dec.workspace.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    assert dec.check() == 7          # MLA_ERR_PLAN_MISMATCH
    dec.workspace.zero_()
    (o2, l2), _ = run_gpu(bt, dev=dev)
    ro, rl = oracle(bt)
    assert_close(o2, l2, ro, rl)


@pytest.mark.parametrize("H,num_sms", [(128, 8), (16, 4)])
def test_many_items_per_worker(H, num_sms):
    # hundreds of short requests on a handful of workers: a worker's items go
    # past the two-CTA kernel's 64-item shared-memory copy (the rest are read
    # from the plan in global memory), with empty and one-token requests mixed in
    rng = np.random.default_rng(2000 + H)
    lengths = [int(x) for x in rng.integers(0, 6, size=700)]
    lengths[5] = 300
    bt = _batch(lengths, H, pool=sum(lengths) + 50, seed=21)
    (out, lse), dec = run_gpu(bt, num_sms=num_sms)
    W = dec.header[6]
    items = dec.header[8]
    assert items / W > 64                        # the fallback is exercised
    ro, rl = oracle(bt)
    assert_close(out, lse, ro, rl)


@pytest.mark.parametrize("H", [16, 128])
def test_rows_past_4_gib_of_the_pool(H):
    # every row the batch reads sits above slot 2^22 of a 4.8 GB pool (byte
    # offsets past 2^32); the result equals the oracle on the compact pool
    # (the slot numbers are only names), and an append past 2^22 lands exactly
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    bt = _batch([300, 5, 1000, 64], H, seed=77 + H)
    dev = to_device(bt)
    base, big = 1 << 22, (1 << 22) + 4096
    used = np.unique(bt.kv_indices)
    assert used.size < big - base
    mapping = np.full(bt.kv_cache.shape[0], -1, dtype=np.int64)
    mapping[used] = base + np.arange(used.size)
    pool = torch.zeros((big, 576), dtype=torch.bfloat16, device="cuda")
    pool[torch.from_numpy(mapping[used]).cuda()] = dev["kv_cache"][torch.from_numpy(used.astype(np.int64)).cuda()]
    moved = dict(dev, kv_cache=pool, kv_indices=torch.from_numpy(mapping[bt.kv_indices].astype(np.int32)).cuda())
    (out, lse), _ = run_gpu(bt, dev=moved)
    ro, rl = oracle(bt)
    assert_close(out, lse, ro, rl)

    rows = torch.randn((2, 576), device="cuda").to(torch.bfloat16)
    slots = torch.tensor([big - 1, base + used.size], dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    binding.append_kv(pool, slots, rows, ws)
    assert binding.check_errors(ws) == 0
    assert torch.equal(pool[big - 1], rows[0]) and torch.equal(pool[base + used.size], rows[1])
