"""GPU parity of a shared-prefix cascade built from the library's calls: a
prefix pass with the G x H query rows of a request group as the heads of one
request (each prefix row gathered once), an ordinary suffix pass per request,
and mla_merge_two_states -- against the oracle's plain decode over each
request's prefix + suffix rows."""
import numpy as np
import pytest

from tests._helpers import ATOL_LSE, ATOL_OUT, RTOL_OUT

pytestmark = pytest.mark.gpu


def _cascade(H, G, prefix_len, suffix_lens, group, seed, out_dtype="f32"):
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    from oracle import mla_oracle as O
    rng = np.random.default_rng(seed)
    pool = prefix_len + sum(suffix_lens) + 37
    kv = W.f32_to_bf16_bits(rng.standard_normal((pool, 576), dtype=np.float32))
    slots = rng.permutation(pool).astype(np.int32)
    prefix = slots[:prefix_len]
    suffix = slots[prefix_len:prefix_len + sum(suffix_lens)]
    s_ptr = np.concatenate([[0], np.cumsum(suffix_lens)]).astype(np.int32)
    qn = W.f32_to_bf16_bits(rng.standard_normal((G, H, 512), dtype=np.float32))
    qr = W.f32_to_bf16_bits(rng.standard_normal((G, H, 64), dtype=np.float32))
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    ti = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    kv_d, qn_d, qr_d = bf(kv), bf(qn), bf(qr)
    o_p = torch.empty((G, H, 512), dtype=torch.float32, device="cuda")
    l_p = torch.empty((G, H), dtype=torch.float32, device="cuda")
    # prefix pass, one group of requests at a time (at most 128 query rows)
    for g0 in range(0, G, group):
        g1 = min(G, g0 + group)
        ptr = np.array([0, prefix_len], dtype=np.int32)
        dec = binding.Decoder(ptr, (g1 - g0) * H)
        dec.run(qn_d[g0:g1], qr_d[g0:g1], kv_d, ti(ptr), ti(prefix), 1.0 / np.sqrt(192.0), o_p[g0:g1], l_p[g0:g1])
        assert dec.check() == 0
    # suffix pass
    o_s = torch.empty((G, H, 512), dtype=torch.float32, device="cuda")
    l_s = torch.empty((G, H), dtype=torch.float32, device="cuda")
    dec = binding.Decoder(s_ptr, H)
    dec.run(qn_d, qr_d, kv_d, ti(s_ptr), ti(suffix if suffix.size else np.zeros(1, np.int32)), 1.0 / np.sqrt(192.0),
            o_s, l_s)
    assert dec.check() == 0
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    out = torch.empty((G, H, 512), dtype=dt, device="cuda")
    lse = torch.empty((G, H), dtype=torch.float32, device="cuda")
    binding.merge_two_states(o_p, l_p, o_s, l_s, out, lse)
    torch.cuda.synchronize()
    # reference: each request over its prefix + suffix rows
    full_ptr = np.concatenate([[0], np.cumsum([prefix_len + n for n in suffix_lens])]).astype(np.int32)
    full_ind = np.concatenate([np.concatenate([prefix, suffix[s_ptr[b]:s_ptr[b + 1]]]) for b in range(G)])
    ro, rl = O.decode_attention(qn, qr, kv, full_ptr, full_ind.astype(np.int32), 1.0 / np.sqrt(192.0))
    o = out.float().cpu().numpy()
    err = np.abs(o - ro)
    assert (err <= ATOL_OUT + RTOL_OUT * np.abs(ro)).all(), f"out: max err {err.max():.3e}"
    assert np.abs(lse.cpu().numpy() - rl).max() <= ATOL_LSE


@pytest.mark.parametrize("H,G,group", [(16, 8, 8), (16, 2, 2), (32, 4, 4), (64, 2, 2), (16, 12, 8)])
def test_shared_prefix_cascade_matches_full_decode(H, G, group):
    rng = np.random.default_rng(H * 100 + G)
    suffix_lens = [int(x) for x in rng.integers(0, 300, size=G)]
    suffix_lens[0] = 0                           # a request with no suffix of its own
    _cascade(H, G, prefix_len=2100, suffix_lens=suffix_lens, group=group, seed=H + G)


def test_cascade_bf16_output_and_in_place_merge():
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    _cascade(16, 4, prefix_len=700, suffix_lens=[5, 64, 129, 1], group=4, seed=3, out_dtype="bf16")
    # in-place: out aliases the first state
    rng = np.random.default_rng(4)
    a = torch.from_numpy(rng.standard_normal((6, 512)).astype(np.float32)).cuda()
    b = torch.from_numpy(rng.standard_normal((6, 512)).astype(np.float32)).cuda()
    la = torch.tensor([0.5, -np.inf, 3.0, -np.inf, 1.0, 2.0], dtype=torch.float32).cuda()
    lb = torch.tensor([1.5, 2.0, -np.inf, -np.inf, 1.0, -5.0], dtype=torch.float32).cuda()
    from oracle import mla_oracle as O
    ref = [O.merge_states(np.stack([a.cpu().numpy()[r:r + 1][:, None], b.cpu().numpy()[r:r + 1][:, None]])[:, 0],
                          np.array([[la[r].item()], [lb[r].item()]])) for r in range(6)]
    binding.merge_two_states(a, la, b, lb, a, la)
    torch.cuda.synchronize()
    for r in range(6):
        np.testing.assert_allclose(a.cpu().numpy()[r], ref[r][0][0], rtol=1e-5, atol=1e-6)
        rl = ref[r][1][0]
        assert (np.isneginf(rl) and np.isneginf(la[r].item())) or abs(la[r].item() - rl) < 1e-5
