"""Shared helpers for the GPU parity tests: move a synthetic batch to the
device, run it through the C ABI, and compare with the fp64 oracle."""
import numpy as np

ATOL_OUT = 1e-2
RTOL_OUT = 1e-2
ATOL_LSE = 2e-3


def to_device(batch, device="cuda"):
    import torch
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return dict(
        q_nope=bf(batch.q_nope), q_rope=bf(batch.q_rope), kv_cache=bf(batch.kv_cache),
        kv_indptr=torch.from_numpy(batch.kv_indptr.astype(np.int32)).to(device),
        kv_indices=torch.from_numpy(batch.kv_indices.astype(np.int32)).to(device),
    )


def run_gpu(batch, out_dtype=None, dev=None, num_sms=0, with_lse=True, repeat=1):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    out_dtype = out_dtype or torch.float32
    dev = dev or to_device(batch)
    dec = binding.Decoder(batch.kv_indptr, batch.heads, num_sms=num_sms)
    B, H = batch.batch, batch.heads
    outs = []
    for _ in range(repeat):
        out = torch.full((B, H, 512), float("nan"), dtype=out_dtype, device="cuda")
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
        dec.run(dev["q_nope"], dev["q_rope"], dev["kv_cache"], dev["kv_indptr"], dev["kv_indices"],
                batch.sm_scale, out, lse)
        st = dec.check()
        assert st == 0, binding.status_string(st)
        outs.append((out.float().cpu().numpy(), None if lse is None else lse.cpu().numpy()))
    return outs if repeat > 1 else outs[0], dec


def oracle(batch, requests=None):
    from oracle import mla_oracle as O
    return O.decode_attention(batch.q_nope, batch.q_rope, batch.kv_cache, batch.kv_indptr, batch.kv_indices,
                              batch.sm_scale, requests=requests)


def assert_close(out, lse, ref_out, ref_lse, requests=None, out_atol=ATOL_OUT, out_rtol=RTOL_OUT):
    rows = slice(None) if requests is None else list(requests)
    o, r = out[rows], ref_out[rows]
    err = np.abs(o - r)
    bound = out_atol + out_rtol * np.abs(r)
    bad = err > bound
    assert not np.isnan(o).any(), "NaN in output"
    assert not bad.any(), f"out mismatch: {bad.sum()} elements, max err {err.max():.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}"
    if lse is not None:
        l, rl = lse[rows], ref_lse[rows]
        fin = np.isfinite(rl)
        assert np.array_equal(np.isfinite(l), fin), "lse finiteness differs"
        assert np.all(np.isneginf(l[~fin])), "empty request lse must be -inf"
        if fin.any():
            e = np.abs(l[fin] - rl[fin])
            assert e.max() <= ATOL_LSE, f"lse mismatch: max err {e.max():.3e}"
