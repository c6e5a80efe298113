"""GPU parity of the per-head products around the decode (mla_absorb_query,
mla_project_output) against the fp64 oracle, and of the whole absorbing path
(absorb -> decode -> project) against the oracle's absorbed attention."""
import numpy as np
import pytest

from tests._helpers import to_device

pytestmark = pytest.mark.gpu


def _bf(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _f64(bits):
    from oracle import mla_oracle as O
    return O.bf16_bits_to_f64(bits)


def _bits(t):
    return t.cpu().view(__import__("torch").int16).numpy().view(np.uint16)


def _check(got, ref, atol, rtol, what):
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert (err <= bound).all(), f"{what}: {int((err > bound).sum())} elements off, max err {err.max():.3e}"


# bf16 results: the kernel's fp32 sum rounded once to bf16 (<= 2^-9 relative)
BF16_ATOL, BF16_RTOL = 2e-3, 4e-3


@pytest.mark.parametrize("B,H", [(1, 16), (5, 32), (64, 16), (130, 128), (200, 48)])
def test_absorb_query_matches_oracle(B, H):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    from oracle import mla_oracle as O
    x = W.make_head_product_inputs(B, H, seed=100 + B + H)
    q = torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    binding.absorb_query(_bf(x.q_pre), _bf(x.w_kc), q)
    torch.cuda.synchronize()
    ref = O.absorb_query(_f64(x.q_pre), _f64(x.w_kc))
    _check(q.float().cpu().numpy(), ref, BF16_ATOL, BF16_RTOL, "absorb")


@pytest.mark.parametrize("B,H,out_dtype", [(1, 16, "f32"), (7, 64, "bf16"), (64, 16, "f32"), (130, 128, "f32"),
                                           (200, 32, "bf16")])
def test_project_output_matches_oracle(B, H, out_dtype):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    from oracle import mla_oracle as O
    x = W.make_head_product_inputs(B, H, seed=200 + B + H)
    rng = np.random.default_rng(300 + B)
    o_lat = W.f32_to_bf16_bits(rng.standard_normal((B, H, 512), dtype=np.float32))
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    out = torch.full((B, H, 128), float("nan"), dtype=dt, device="cuda")
    binding.project_output(_bf(o_lat), _bf(x.w_vc), out)
    torch.cuda.synchronize()
    ref = O.project_output(_f64(o_lat), _f64(x.w_vc))
    if out_dtype == "f32":
        _check(out.cpu().numpy(), ref, 1e-4, 1e-4, "project fp32")
    else:
        _check(out.float().cpu().numpy(), ref, BF16_ATOL, BF16_RTOL, "project bf16")


@pytest.mark.parametrize("H", [16, 128])
def test_absorbing_path_end_to_end(H):
    # q_pre -> absorb (bf16) -> decode (bf16 latent output) -> project (fp32)
    # on the GPU; each stage checked against the oracle, which takes its own
    # inputs (never the GPU's intermediate results): the absorbed query and
    # the decode output as the oracle computes them, rounded to bf16 where the
    # GPU path rounds; then the whole chain against the oracle's fp64
    # absorbed attention
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    from oracle import mla_oracle as O
    lengths = [1, 40, 257, 700]
    bt = W.make_batch(lengths, heads=H, pool=2048, seed=41 + H)
    x = W.make_head_product_inputs(bt.batch, H, seed=42 + H)
    dev = to_device(bt)
    q_lat = torch.empty((bt.batch, H, 512), dtype=torch.bfloat16, device="cuda")
    binding.absorb_query(_bf(x.q_pre), _bf(x.w_kc), q_lat)
    dec = binding.Decoder(bt.kv_indptr, H)
    o_lat = torch.empty((bt.batch, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((bt.batch, H), dtype=torch.float32, device="cuda")
    dec.run(q_lat, dev["q_rope"], dev["kv_cache"], dev["kv_indptr"], dev["kv_indices"], bt.sm_scale, o_lat, lse)
    out = torch.empty((bt.batch, H, 128), dtype=torch.float32, device="cuda")
    binding.project_output(o_lat, _bf(x.w_vc), out)
    assert dec.check() == 0
    q_bits, o_bits = _bits(q_lat), _bits(o_lat)
    # stage by stage, each oracle stage on the oracle's previous stage
    q_ref = O.absorb_query(_f64(x.q_pre), _f64(x.w_kc))
    _check(_f64(q_bits), q_ref, BF16_ATOL, BF16_RTOL, "absorb")
    q_ref_bits = W.f32_to_bf16_bits(q_ref.astype(np.float32))
    ro, _ = O.decode_attention(q_ref_bits, bt.q_rope, bt.kv_cache, bt.kv_indptr, bt.kv_indices, bt.sm_scale)
    _check(_f64(o_bits), ro, 1e-2, 1e-2, "decode")
    o_ref_bits = W.f32_to_bf16_bits(ro.astype(np.float32))
    p_ref = O.project_output(_f64(o_ref_bits), _f64(x.w_vc))
    # the GPU projects its own bf16 decode output: within the decode bar of
    # o, carried through w_vc (gain 1), plus the fp32 sum's rounding
    _check(out.cpu().numpy(), p_ref, 2e-2, 2e-2, "project")
    # whole chain against the fp64 absorbing path of each request
    for b, L in enumerate(lengths):
        rows = O.gather_rows(bt.kv_cache, bt.kv_indices, int(bt.kv_indptr[b]), int(bt.kv_indptr[b + 1]))
        q_lat_ref = O.absorb_query(_f64(x.q_pre)[b:b + 1], _f64(x.w_kc))[0]
        o_ref, _ = O.partial_state(q_lat_ref, _f64(bt.q_rope[b]), rows, bt.sm_scale)
        ref = O.project_output(o_ref[None], _f64(x.w_vc))[0]
        _check(out.cpu().numpy()[b], ref, 2e-2, 2e-2, f"chain request {b}")
