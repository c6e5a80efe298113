"""The workspace-free entry point (mla_decode_run_noalloc), for callers that
cannot allocate device memory: its output must match mla_decode_run's on the
same plan, call after call.  Kept in a file of its own that pytest collects
last, so a failure here comes after every other test has run."""
import numpy as np
import pytest

from tests._helpers import assert_close, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,lengths", [(16, [20000, 3, 700]), (128, [9000, 65, 1])])
def test_noalloc_matches_run_two_calls_in_a_row(H, lengths):
    import torch
    from mla_latent_kv_absorbed_gb300 import build
    build.build()
    from mla_latent_kv_absorbed_gb300 import binding
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
    ro, rl = ref_out.cpu().numpy().astype(np.float64), ref_lse.cpu().numpy().astype(np.float64)
    for _ in range(2):
        out = torch.full((B, H, 512), float("nan"), device="cuda")
        lse = torch.full((B, H), float("nan"), device="cuda")
        binding.decode_run_noalloc(dec.plan_host, dec.plan_dev, dev["q_nope"], dev["q_rope"], dev["kv_cache"],
                                   dev["kv_indptr"], dev["kv_indices"], bt.sm_scale, out, lse)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), lse.cpu().numpy(), ro, rl)


def test_noalloc_rejects_plans_beyond_its_buffer():
    from mla_latent_kv_absorbed_gb300 import build
    build.build()
    from mla_latent_kv_absorbed_gb300 import binding
    # a long request cut over 500 workers at H=128 needs ~130 MB of partial
    # states, far beyond the fixed buffer; the call must refuse on the host
    plan, ws = binding.decode_plan(np.array([0, 200000], dtype=np.int32), 128, num_sms=1000)
    assert ws > binding.NOALLOC_SCRATCH_BYTES
    lib = binding.library()
    st = lib.mla_decode_run_noalloc(np.ascontiguousarray(plan).ctypes.data, 1 << 20, 1 << 20, 1 << 20, 1 << 20,
                                    1000, 1 << 20, 1 << 20, 0.1, 1 << 20, 0, None, None)
    assert st == 3                                  # MLA_ERR_WORKSPACE, nothing launched
