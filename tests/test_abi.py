"""Host-side tests of the C ABI (no GPU needed): the library loads, exports
every entry point include/*.h declares, its plan matches the restatement in
oracle/plan_ref.py word for word, and bad arguments are rejected on the host
before any launch."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from mla_latent_kv_absorbed_gb300 import build
    build.build()
    from mla_latent_kv_absorbed_gb300 import binding
    return binding


_FAKE = {}


def _fake_ptr():
    """A device address for the rejection tests.  Every case below must fail
    its host check before any launch; should a check regress, what a kernel
    would get is a zero-filled 16 MiB device buffer when a GPU is present
    (every pointer below, with its small offsets, stays inside it), and on a
    machine without a GPU nothing can launch at all."""
    if "p" not in _FAKE:
        try:
            import torch
            have = torch.cuda.is_available()
        except Exception:
            have = False
        if have:
            _FAKE["buf"] = torch.zeros(16 << 20, dtype=torch.uint8, device="cuda")
            _FAKE["p"] = int(_FAKE["buf"].data_ptr())
        else:
            _FAKE["p"] = 1 << 20
    return _FAKE["p"]


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(mla_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(B):
    declared = _declared_functions()
    assert "mla_decode_run" in declared and "mla_decode_plan" in declared
    lib = B.library()
    for name in declared:
        assert hasattr(lib, name), name
    assert set(B.EXPORTS) <= set(declared)
    assert B.abi_version() == 1


def test_status_strings(B):
    for code, name in B.STATUS_NAMES.items():
        assert B.status_string(code) == name
    assert B.status_string(99) == "MLA_ERR_UNKNOWN"


def _cases():
    rng = np.random.default_rng(5)
    out = [([0], 16), ([0, 0, 0], 128), ([0, 1], 16), ([0, 1], 128), ([0, 131072], 128),
           ([0, 65536, 196608], 128), ([0, 7, 7, 40, 2000], 32), ([0, 4096] * 1, 64)]
    for H in (16, 32, 48, 64, 96, 112, 128):
        for _ in range(6):
            Bn = int(rng.integers(1, 260))
            L = rng.integers(0, 6000, size=Bn)
            if rng.random() < 0.4:
                L[rng.integers(0, Bn)] = int(rng.integers(30000, 140000))
            out.append((np.concatenate([[0], np.cumsum(L)]).tolist(), H))
    return out


@pytest.mark.parametrize("sms", [152, 148, 7])
def test_plan_matches_restatement_bit_exact(B, sms):
    from oracle import plan_ref as PR
    for indptr, H in _cases():
        words, ws = B.decode_plan(np.asarray(indptr, dtype=np.int32), H, num_sms=sms)
        ref_words, ref_ws = PR.build_plan(indptr, H, sms)
        assert words.tolist() == ref_words, (indptr[:5], H)
        assert ws == ref_ws


def test_plan_workloads_bit_exact(B):
    from oracle import plan_ref as PR
    from mla_latent_kv_absorbed_gb300 import workloads as W
    for n, spec in W.WORKLOADS.items():
        rng = np.random.default_rng(spec.seed)
        L = W.draw_lengths(spec, rng)
        indptr = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
        words, ws = B.decode_plan(indptr, spec.heads, num_sms=152)
        ref, ref_ws = PR.build_plan(indptr.tolist(), spec.heads, 152)
        assert words.tolist() == ref and ws == ref_ws


def _plan_raw(B, indptr, H, sms=152, plan_words=None):
    lib = B.library()
    arr = np.ascontiguousarray(indptr, dtype=np.int32)
    need, ws = ctypes.c_size_t(0), ctypes.c_size_t(0)
    buf = None if plan_words is None else np.zeros(plan_words, dtype=np.int32)
    st = lib.mla_decode_plan(arr.ctypes.data, arr.shape[0] - 1, H, sms,
                             None if buf is None else buf.ctypes.data, 0 if buf is None else plan_words,
                             ctypes.byref(need), ctypes.byref(ws))
    return st, need.value, ws.value


def test_plan_rejects_bad_input(B):
    assert _plan_raw(B, [1, 5], 16)[0] == 1            # indptr[0] != 0
    assert _plan_raw(B, [0, 5, 3], 16)[0] == 1         # decreasing
    assert _plan_raw(B, [0, 5], 8)[0] == 2             # unsupported heads
    assert _plan_raw(B, [0, 5], 136)[0] == 2
    assert _plan_raw(B, [0, 5], 16, sms=-1)[0] == 1
    st, need, _ = _plan_raw(B, [0, 5, 9], 16)
    assert st == 0 and need > 16
    st2, need2, _ = _plan_raw(B, [0, 5, 9], 16, plan_words=need - 1)
    assert st2 == 3 and need2 == need                   # too small, size still reported
    lib = B.library()
    assert lib.mla_decode_plan(None, 1, 16, 152, None, 0, None, None) == 1


def test_run_rejects_bad_arguments_before_launch(B):
    lib = B.library()
    plan, ws_bytes = B.decode_plan(np.array([0, 100, 300], dtype=np.int32), 16, num_sms=152)
    fake = _fake_ptr()   # never dereferenced: every case below fails its host check first

    def run(plan_host=plan, plan_dev=fake, ws=fake, ws_bytes=ws_bytes, out_dtype=0, slots=1000, q=fake,
            scale=0.1):
        ph = None if plan_host is None else np.ascontiguousarray(plan_host, dtype=np.int32)
        return lib.mla_decode_run(None if ph is None else ph.ctypes.data, plan_dev, q, fake, fake, slots,
                                  fake, fake, ctypes.c_float(scale), fake, out_dtype, fake, ws, ws_bytes,
                                  None)

    assert run(plan_host=None) == 1
    bad = plan.copy(); bad[0] = 0
    assert run(plan_host=bad) == 1                       # magic
    bad = plan.copy(); bad[13] += 1
    assert run(plan_host=bad) == 1                       # word count
    assert run(plan_dev=None) == 1
    assert run(out_dtype=3) == 2
    assert run(ws=None) == 1
    assert run(ws=fake + 4) == 1                         # misaligned workspace
    assert run(ws_bytes=0) == 3 if plan[9] > 0 else True
    assert run(slots=0) == 1
    assert run(q=fake + 2) == 1                          # misaligned q_nope
    assert run(scale=float("nan")) == 1


def test_tree_run_rejects_bad_arguments_before_launch(B):
    # draft trees: width, head multiple, parents and mask scratch are checked
    # on the host before the mask kernel or the decode is launched
    lib = B.library()
    fake = _fake_ptr()
    plan, ws_bytes = B.decode_plan(np.array([0, 100, 300], dtype=np.int32), 16 * 4, num_sms=152)
    ph = np.ascontiguousarray(plan, dtype=np.int32)

    def run(W=4, parents=fake, masks=fake):
        return lib.mla_decode_run_tree(ph.ctypes.data, fake, W, parents, masks, fake, fake, fake, 1000, fake, fake,
                                       ctypes.c_float(0.1), fake, 0, fake, fake, ws_bytes, None)

    assert run(W=0) == 1
    assert run(W=3) == 1                                 # 64 rows are not a multiple of 3
    assert run(parents=None) == 1
    assert run(masks=None) == 1
    assert run(masks=fake + 4) == 1                      # mask words are 8-byte aligned
    assert run(parents=fake + 2) == 1
    plan128, ws128 = B.decode_plan(np.array([0, 100], dtype=np.int32), 128, num_sms=152)
    ph128 = np.ascontiguousarray(plan128, dtype=np.int32)
    assert lib.mla_decode_run_tree(ph128.ctypes.data, fake, 128, fake, fake, fake, fake, fake, 1000, fake, fake,
                                   ctypes.c_float(0.1), fake, 0, fake, fake, ws128, None) == 2   # W > 64


def test_merge_rejects_bad_arguments(B):
    lib = B.library()
    assert lib.mla_merge_states(None, None, None, -1, 16, None, 0, None, None) == 1
    assert lib.mla_merge_states(None, None, None, 2, 16, None, 5, None, None) == 2
    assert lib.mla_merge_states(None, None, None, 2, 16, None, 0, None, None) == 1
    assert lib.mla_merge_states(None, None, None, 0, 16, None, 0, None, None) == 0
    assert lib.mla_check_errors(None, None) == 1


def test_head_products_reject_bad_arguments(B):
    lib = B.library()
    fake = _fake_ptr()
    # unsupported head dims, then bad sizes and pointers; all before any launch
    assert lib.mla_absorb_query(fake, fake, fake, 4, 16, 64, None, None) == 2
    assert lib.mla_absorb_query(fake, fake, fake, -1, 16, 128, None, None) == 1
    assert lib.mla_absorb_query(fake, fake, fake, 4, 0, 128, None, None) == 1
    assert lib.mla_absorb_query(None, fake, fake, 4, 16, 128, None, None) == 1
    assert lib.mla_absorb_query(fake + 2, fake, fake, 4, 16, 128, None, None) == 1
    assert lib.mla_absorb_query(fake, fake, fake, 4, 16, 128, fake + 4, None) == 1
    assert lib.mla_absorb_query(None, None, None, 0, 16, 128, None, None) == 0
    assert lib.mla_project_output(fake, fake, fake, 0, 4, 16, 96, None, None) == 2
    assert lib.mla_project_output(fake, fake, fake, 3, 4, 16, 128, None, None) == 2
    assert lib.mla_project_output(fake, fake, fake, 0, -2, 16, 128, None, None) == 1
    assert lib.mla_project_output(fake, None, fake, 1, 4, 16, 128, None, None) == 1
    assert lib.mla_project_output(fake, fake, fake + 8, 0, 4, 16, 128, None, None) == 1
    assert lib.mla_project_output(None, None, None, 0, 0, 16, 128, None, None) == 0


def test_append_rejects_bad_arguments(B):
    lib = B.library()
    fake = _fake_ptr()
    assert lib.mla_append_kv(fake, 100, fake, fake, -1, None, None) == 1
    assert lib.mla_append_kv(fake, 0, fake, fake, 2, None, None) == 1
    assert lib.mla_append_kv(None, 100, fake, fake, 2, None, None) == 1
    assert lib.mla_append_kv(fake, 100, fake, fake + 8, 2, None, None) == 1
    assert lib.mla_append_kv(None, 100, None, None, 0, None, None) == 0


def test_wait_probe_rejects_bad_arguments(B):
    lib = B.library()
    lib.mla_probe_wait_limit.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    fake = _fake_ptr()
    assert lib.mla_probe_wait_limit(None, None) == 1
    assert lib.mla_probe_wait_limit(fake + 4, None) == 1


def test_merge_two_rejects_bad_arguments(B):
    lib = B.library()
    fake = _fake_ptr()
    assert lib.mla_merge_two_states(fake, fake, fake, fake, 4, fake, 2, None, None) == 2
    assert lib.mla_merge_two_states(fake, fake, fake, fake, -1, fake, 0, None, None) == 1
    assert lib.mla_merge_two_states(None, fake, fake, fake, 4, fake, 0, None, None) == 1
    assert lib.mla_merge_two_states(fake + 4, fake, fake, fake, 4, fake, 0, None, None) == 1
    assert lib.mla_merge_two_states(None, None, None, None, 0, None, 0, None, None) == 0


def test_fp8_entry_points_reject_bad_arguments(B):
    lib = B.library()
    fake = _fake_ptr()
    plan, ws_bytes = B.decode_plan(np.array([0, 100, 300], dtype=np.int32), 16, num_sms=152)
    need = B.decode_fp8_workspace_bytes(plan)
    # plan workspace + two 18 KB query images + 2 x 16 factors, 256-byte aligned regions
    assert need >= ws_bytes + 2 * 4 * 16 * 288 + 2 * 16 * 4
    plan128, ws128 = B.decode_plan(np.array([0, 100], dtype=np.int32), 128, num_sms=152)
    assert B.decode_fp8_workspace_bytes(plan128) >= ws128     # the two-CTA kernel reads FP8 too
    n = ctypes.c_size_t(0)
    assert lib.mla_decode_fp8_workspace_bytes(None, ctypes.byref(n)) == 1

    def run(plan_host=plan, kv_scale=0.03125, ws=fake, wsb=need, out_dtype=0, q=fake, slots=1000, scale=0.1):
        ph = np.ascontiguousarray(plan_host, dtype=np.int32)
        return lib.mla_decode_run_fp8(ph.ctypes.data, fake, q, fake, fake, slots, ctypes.c_float(kv_scale), fake,
                                      fake, ctypes.c_float(scale), fake, out_dtype, fake, ws, wsb, None)

    assert run(kv_scale=0.0) == 1 and run(kv_scale=-1.0) == 1 and run(kv_scale=float("inf")) == 1
    assert run(scale=float("nan")) == 1
    assert run(out_dtype=2) == 2
    assert run(wsb=need - 1) == 3                        # the plan's workspace alone is not enough
    assert run(ws=fake + 8) == 1
    assert run(q=fake + 2) == 1
    assert run(slots=0) == 1
    assert lib.mla_append_kv_fp8(fake, 100, fake, fake, 2, ctypes.c_float(0.0), None, None) == 1
    assert lib.mla_append_kv_fp8(fake, 100, fake, fake, -1, ctypes.c_float(1.0), None, None) == 1
    assert lib.mla_append_kv_fp8(fake + 4, 100, fake, fake, 2, ctypes.c_float(1.0), None, None) == 1
    assert lib.mla_append_kv_fp8(None, 100, None, None, 0, ctypes.c_float(1.0), None, None) == 0


def test_graph_capacities_hold_every_plan_they_promise(B):
    # any plan for batch <= max_batch (same heads and SMs) fits the capacities of mla_decode_graph_sizes
    rng = np.random.default_rng(12)
    for H, sms, max_batch in ((16, 152, 40), (128, 152, 24), (32, 20, 9), (64, 7, 5)):
        words, ws = B.decode_graph_sizes(max_batch, H, sms)
        for _ in range(60):
            b = int(rng.integers(0, max_batch + 1))
            kind = rng.integers(0, 3)
            if kind == 0:
                lens = rng.integers(0, 5000, size=b)
            elif kind == 1:
                lens = np.full(b, int(rng.integers(1, 70000)))
            else:
                lens = np.where(rng.random(b) < 0.5, 0, rng.integers(1, 300, size=b))
            indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
            plan, need_ws = B.decode_plan(indptr, H, num_sms=sms)
            assert plan.size <= words and need_ws <= ws, (H, sms, b)
    lib = B.library()
    n = ctypes.c_size_t(0)
    assert lib.mla_decode_graph_sizes(0, 16, 152, ctypes.byref(n), None) == 1
    assert lib.mla_decode_graph_sizes(4, 16, 0, ctypes.byref(n), None) == 1
    assert lib.mla_decode_graph_sizes(4, 24, 152, ctypes.byref(n), None) == 2


def test_graph_run_rejects_bad_arguments(B):
    lib = B.library()
    fake = _fake_ptr()
    words, ws = B.decode_graph_sizes(8, 16, 152)

    def run(pw=words, wsb=ws, q=fake, heads=16, out_dtype=0, plan=fake):
        return lib.mla_decode_run_graph(plan, pw, 8, heads, 152, q, fake, fake, 1000, fake, fake, ctypes.c_float(0.1),
                                        fake, out_dtype, fake, fake, wsb, None)

    assert run(pw=words - 1) == 3 and run(wsb=ws - 1) == 3
    assert run(q=fake + 2) == 1 and run(plan=None) == 1
    assert run(heads=24) == 2 and run(out_dtype=5) == 2


def test_binding_refuses_to_load_without_the_library(tmp_path):
    # the binding has no fallback: beside no built library, importing it raises
    import importlib.util
    import shutil
    src = os.path.join(ROOT, "mla_latent_kv_absorbed_gb300", "binding.py")
    shutil.copy(src, tmp_path / "binding.py")
    spec = importlib.util.spec_from_file_location("mla_binding_without_library", tmp_path / "binding.py")
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError, match="libmla_decode.so is missing"):
        spec.loader.exec_module(mod)


def test_empty_batch_run_checks_arguments_and_launches_nothing(B):
    # batch == 0: the host checks still apply to the plan, plan_dev and the
    # workspace; the data pointers may be NULL and no CUDA call is made
    lib = B.library()
    plan, ws_bytes = B.decode_plan(np.array([0], dtype=np.int32), 16, num_sms=152)
    assert plan[2] == 0
    fake = _fake_ptr()   # never dereferenced
    ph = np.ascontiguousarray(plan, dtype=np.int32)

    def run(plan_dev=fake, ws=fake):
        return lib.mla_decode_run(ph.ctypes.data, plan_dev, None, None, None, 1, None, None, ctypes.c_float(0.1),
                                  None, 0, None, ws, ws_bytes, None)

    assert run() == 0
    assert run(plan_dev=None) == 1
    assert run(ws=None) == 1


def test_wrappers_refuse_index_arrays_shorter_than_the_plan(B):
    # the kernels trust kv_indices to hold the slots kv_indptr names (the ABI
    # passes no lengths): every binding wrapper with a host plan checks both
    # sizes against the plan before any launch
    import torch
    plan, _ = B.decode_plan(np.array([0, 100, 300], dtype=np.int32), 16, num_sms=152)
    assert B.plan_nnz(plan) == 300
    ok_ptr, ok_idx = torch.zeros(3, dtype=torch.int32), torch.zeros(300, dtype=torch.int32)
    B._check_csr(plan, ok_ptr, ok_idx, "t")
    with pytest.raises(ValueError, match="kv_indices has 299 entries"):
        B._check_csr(plan, ok_ptr, torch.zeros(299, dtype=torch.int32), "t")
    with pytest.raises(ValueError, match="kv_indptr has 4 entries"):
        B._check_csr(plan, torch.zeros(4, dtype=torch.int32), ok_idx, "t")
    # the wrappers raise before touching the library (CPU tensors stand in)
    x = torch.zeros(4, dtype=torch.float32)
    short = torch.zeros(299, dtype=torch.int32)
    for call in (lambda: B.decode_run(plan, x, x, x, x, ok_ptr, short, 0.1, x, None, x),
                 lambda: B.decode_attend(plan, x, x, x, x, ok_ptr, short, 0.1, x, None, x),
                 lambda: B.decode_run_noalloc(plan, x, x, x, x, ok_ptr, short, 0.1, x, None),
                 lambda: B.decode_run_fp8(plan, x, x, x, x, 0.03, ok_ptr, short, 0.1, x, None, x),
                 lambda: B.decode_run_multi_query(plan, x, 1, x, x, x, ok_ptr, short, 0.1, x, None, x),
                 lambda: B.decode_run_tree(plan, x, torch.zeros((2, 1), dtype=torch.int32),
                                           torch.zeros((2, 1), dtype=torch.int64), x, x, x, ok_ptr, short, 0.1, x,
                                           None, x)):
        with pytest.raises(ValueError, match="kv_indices has 299 entries"):
            call()
    # an empty batch covers no tokens
    empty, _ = B.decode_plan(np.array([0], dtype=np.int32), 16, num_sms=152)
    assert B.plan_nnz(empty) == 0
