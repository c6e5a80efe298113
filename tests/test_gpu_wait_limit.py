"""Failure handling without a GPU fault: every device-side wait of the kernels
is bounded, and a wait that runs out ends as MLA_ERR_TIMEOUT in the workspace
status word, with the context still usable.  mla_probe_wait_limit runs that
same bounded wait on a barrier that nothing completes; the test checks the
status the host reads, the time the wait took, and that a decode launched
right after it matches the oracle and reports no error."""
import time

import numpy as np
import pytest

from tests._helpers import assert_close, oracle, to_device

pytestmark = pytest.mark.gpu

MLA_ERR_TIMEOUT = 5


def _binding():
    from mla_latent_kv_absorbed_gb300 import build
    build.build()
    from mla_latent_kv_absorbed_gb300 import binding
    return binding


def test_wait_that_nothing_completes_times_out_and_context_survives():
    import torch
    binding = _binding()
    from mla_latent_kv_absorbed_gb300 import workloads as W

    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    binding.probe_wait_limit(ws)
    st = binding.check_errors(ws)                  # synchronises, reads and clears
    dt = time.perf_counter() - t0
    assert st == MLA_ERR_TIMEOUT
    assert 0.5 < dt < 30.0                         # the limit is about 1 s of wall time
    assert binding.check_errors(ws) == 0           # cleared by the read

    # the context is intact: a decode right after is correct and clean
    H, lengths = 16, [700, 3, 129]
    bt = W.make_batch(lengths, heads=H, pool=int(np.sum(lengths)) + 64, seed=7)
    dev = to_device(bt)
    dec = binding.Decoder(bt.kv_indptr, H)
    out = torch.empty((bt.batch, H, 512), device="cuda")
    lse = torch.empty((bt.batch, H), device="cuda")
    dec.run(dev["q_nope"], dev["q_rope"], dev["kv_cache"], dev["kv_indptr"], dev["kv_indices"], bt.sm_scale, out, lse)
    assert dec.check() == 0
    oo, ol = oracle(bt)
    assert_close(out.cpu().numpy(), lse.cpu().numpy(), oo, ol)
