"""The workspace-free entry point (mla_decode_run_noalloc), for callers that
cannot allocate device memory while they run a decode step (a memory arena
owned by another runtime, a plugin that only receives tensors).  Its results
must match the fp64 oracle and mla_decode_run's on the same plan, call after
call, and its device status must be readable through
mla_noalloc_check_errors.  Kept in a file of its own that pytest collects
last, so a failure here comes after every other test has run."""
import numpy as np
import pytest

from tests._helpers import assert_close, oracle, to_device

pytestmark = pytest.mark.gpu


def _binding():
    from mla_latent_kv_absorbed_gb300 import build
    build.build()
    from mla_latent_kv_absorbed_gb300 import binding
    return binding


@pytest.mark.parametrize("H,lengths", [(16, [20000, 3, 700]), (128, [9000, 65, 1])])
def test_noalloc_matches_oracle_and_run_two_calls_in_a_row(H, lengths):
    import torch
    binding = _binding()
    from mla_latent_kv_absorbed_gb300 import workloads as W

    bt = W.make_batch(lengths, heads=H, pool=int(np.sum(lengths)) + 64, seed=99)
    dev = to_device(bt)
    dec = binding.Decoder(bt.kv_indptr, H)
    assert dec.header[9] > 0                       # the plan uses partial states (scratch)
    B = bt.batch
    ref_out = torch.empty((B, H, 512), device="cuda")
    ref_lse = torch.empty((B, H), device="cuda")
    dec.run(dev["q_nope"], dev["q_rope"], dev["kv_cache"], dev["kv_indptr"], dev["kv_indices"], bt.sm_scale,
            ref_out, ref_lse)
    assert dec.check() == 0
    run_out, run_lse = ref_out.cpu().numpy(), ref_lse.cpu().numpy()
    oo, ol = oracle(bt)
    assert binding.noalloc_check_errors() == 0     # nothing recorded before the first call
    for _ in range(2):
        out = torch.full((B, H, 512), float("nan"), device="cuda")
        lse = torch.full((B, H), float("nan"), device="cuda")
        binding.decode_run_noalloc(dec.plan_host, dec.plan_dev, dev["q_nope"], dev["q_rope"], dev["kv_cache"],
                                   dev["kv_indptr"], dev["kv_indices"], bt.sm_scale, out, lse)
        assert binding.noalloc_check_errors() == 0
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        assert_close(o, l, oo, ol)                 # the oracle, at the parity tolerance
        assert_close(o, l, run_out, run_lse)       # and the workspace entry point's result


def test_noalloc_status_reports_a_bad_slot_then_clears():
    import torch
    binding = _binding()
    from mla_latent_kv_absorbed_gb300 import workloads as W

    bt = W.make_batch([3000, 40], heads=16, pool=3100, seed=5)
    bt.kv_indices[7] = bt.pool + 100               # out of range: read as row 0 and reported
    dev = to_device(bt)
    dec = binding.Decoder(bt.kv_indptr, 16)
    out = torch.empty((bt.batch, 16, 512), device="cuda")
    binding.decode_run_noalloc(dec.plan_host, dec.plan_dev, dev["q_nope"], dev["q_rope"], dev["kv_cache"],
                               dev["kv_indptr"], dev["kv_indices"], bt.sm_scale, out, None)
    assert binding.noalloc_check_errors() == 6     # MLA_ERR_INDEX_OOB
    assert binding.noalloc_check_errors() == 0     # read and cleared


def test_noalloc_rejects_plans_beyond_its_buffer():
    import ctypes
    import torch
    binding = _binding()
    # a long request cut over 500 workers at H=128 needs ~130 MB of partial
    # states, far beyond the fixed buffer; the call must refuse on the host
    plan, ws = binding.decode_plan(np.array([0, 200000], dtype=np.int32), 128, num_sms=1000)
    assert ws > binding.NOALLOC_SCRATCH_BYTES
    # real (small, zero-filled) device buffers: the call must refuse before any
    # launch, and should that check ever regress a kernel would still only see
    # valid memory
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    lib = binding.library()
    st = lib.mla_decode_run_noalloc(np.ascontiguousarray(plan).ctypes.data, p, p, p, p, 1000, p, p,
                                    ctypes.c_float(0.1), p, 0, None, None)
    assert st == 3                                  # MLA_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert binding.noalloc_check_errors() == 0
