"""Thin ctypes binding of libmla_decode.so (include/mla_decode.h).

Argument marshalling only: every step of the decode path runs in the
library's kernels.  torch is used for device memory and streams.  Importing
this module loads the library and raises if it has not been built (there is
no fallback path).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla_decode.so")

MLA_OK = 0
STATUS_NAMES = {
    0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_WORKSPACE",
    4: "MLA_ERR_CUDA", 5: "MLA_ERR_TIMEOUT", 6: "MLA_ERR_INDEX_OOB", 7: "MLA_ERR_PLAN_MISMATCH",
    8: "MLA_ERR_TREE",
}
EXPORTS = ("mla_status_string", "mla_abi_version", "mla_decode_plan", "mla_decode_run",
           "mla_decode_attend", "mla_decode_merge", "mla_merge_states", "mla_check_errors",
           "mla_decode_run_noalloc", "mla_absorb_query", "mla_project_output",
           "mla_append_kv", "mla_step_staging_bytes", "mla_decode_step_host", "mla_decode_run_multi_query",
           "mla_merge_two_states", "mla_decode_fp8_workspace_bytes", "mla_decode_run_fp8", "mla_append_kv_fp8",
           "mla_decode_graph_sizes", "mla_decode_run_graph", "mla_noalloc_check_errors", "mla_decode_run_tree",
           "mla_probe_wait_limit")
NOALLOC_SCRATCH_BYTES = 32 << 20

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with mla_latent_kv_absorbed_gb300.build.build()")

_lib = ctypes.CDLL(LIB_PATH)
_c_i32p = ctypes.POINTER(ctypes.c_int32)
_c_szp = ctypes.POINTER(ctypes.c_size_t)
_vp = ctypes.c_void_p

_lib.mla_status_string.restype = ctypes.c_char_p
_lib.mla_status_string.argtypes = [ctypes.c_int]
_lib.mla_abi_version.restype = ctypes.c_int
_lib.mla_decode_plan.restype = ctypes.c_int
_lib.mla_decode_plan.argtypes = [_vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp,
                                 ctypes.c_size_t, _c_szp, _c_szp]
_lib.mla_decode_run.restype = ctypes.c_int
_lib.mla_decode_run.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_int64, _vp, _vp, ctypes.c_float,
                                _vp, ctypes.c_int32, _vp, _vp, ctypes.c_size_t, _vp]
_lib.mla_decode_attend.restype = ctypes.c_int
_lib.mla_decode_attend.argtypes = _lib.mla_decode_run.argtypes
_lib.mla_decode_merge.restype = ctypes.c_int
_lib.mla_decode_merge.argtypes = [_vp, _vp, _vp, ctypes.c_int32, _vp, _vp, ctypes.c_size_t, _vp]
_lib.mla_merge_states.restype = ctypes.c_int
_lib.mla_merge_states.argtypes = [_vp, _vp, _vp, ctypes.c_int32, ctypes.c_int32, _vp, ctypes.c_int32,
                                  _vp, _vp]
_lib.mla_decode_run_noalloc.restype = ctypes.c_int
_lib.mla_decode_run_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_int64, _vp, _vp, ctypes.c_float, _vp,
                                        ctypes.c_int32, _vp, _vp]
_lib.mla_check_errors.restype = ctypes.c_int
_lib.mla_check_errors.argtypes = [_vp, _vp]
_lib.mla_noalloc_check_errors.restype = ctypes.c_int
_lib.mla_noalloc_check_errors.argtypes = [_vp]
_lib.mla_probe_wait_limit.restype = ctypes.c_int
_lib.mla_probe_wait_limit.argtypes = [_vp, _vp]
_lib.mla_absorb_query.restype = ctypes.c_int
_lib.mla_absorb_query.argtypes = [_vp, _vp, _vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp, _vp]
_lib.mla_decode_run_multi_query.restype = ctypes.c_int
_lib.mla_decode_run_multi_query.argtypes = [_vp, _vp, ctypes.c_int32, _vp, _vp, _vp, ctypes.c_int64, _vp, _vp,
                                            ctypes.c_float, _vp, ctypes.c_int32, _vp, _vp, ctypes.c_size_t, _vp]
_lib.mla_decode_run_tree.restype = ctypes.c_int
_lib.mla_decode_run_tree.argtypes = [_vp, _vp, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp, ctypes.c_int64, _vp, _vp,
                                     ctypes.c_float, _vp, ctypes.c_int32, _vp, _vp, ctypes.c_size_t, _vp]
_lib.mla_merge_two_states.restype = ctypes.c_int
_lib.mla_merge_two_states.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int64, _vp, ctypes.c_int32, _vp, _vp]
_lib.mla_step_staging_bytes.restype = ctypes.c_size_t
_lib.mla_step_staging_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int32]
_lib.mla_decode_step_host.restype = ctypes.c_int
_lib.mla_decode_step_host.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int32, ctypes.c_int32, _vp, ctypes.c_int64,
                                      ctypes.c_float, _vp, ctypes.c_int32, _vp, _vp, ctypes.c_size_t, _vp,
                                      ctypes.c_size_t, _vp, ctypes.c_size_t, _vp, _vp, _vp]
_lib.mla_append_kv.restype = ctypes.c_int
_lib.mla_append_kv.argtypes = [_vp, ctypes.c_int64, _vp, _vp, ctypes.c_int32, _vp, _vp]
_lib.mla_decode_fp8_workspace_bytes.restype = ctypes.c_int
_lib.mla_decode_fp8_workspace_bytes.argtypes = [_vp, _c_szp]
_lib.mla_decode_run_fp8.restype = ctypes.c_int
_lib.mla_decode_run_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_int64, ctypes.c_float, _vp, _vp,
                                    ctypes.c_float, _vp, ctypes.c_int32, _vp, _vp, ctypes.c_size_t, _vp]
_lib.mla_append_kv_fp8.restype = ctypes.c_int
_lib.mla_append_kv_fp8.argtypes = [_vp, ctypes.c_int64, _vp, _vp, ctypes.c_int32, ctypes.c_float, _vp, _vp]
_lib.mla_decode_graph_sizes.restype = ctypes.c_int
_lib.mla_decode_graph_sizes.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _c_szp, _c_szp]
_lib.mla_decode_run_graph.restype = ctypes.c_int
_lib.mla_decode_run_graph.argtypes = [_vp, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp, _vp,
                                      _vp, ctypes.c_int64, _vp, _vp, ctypes.c_float, _vp, ctypes.c_int32, _vp, _vp,
                                      ctypes.c_size_t, _vp]
_lib.mla_project_output.restype = ctypes.c_int
_lib.mla_project_output.argtypes = [_vp, _vp, _vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                    _vp, _vp]


class MLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


def status_string(status: int) -> str:
    return _lib.mla_status_string(int(status)).decode()


def abi_version() -> int:
    return int(_lib.mla_abi_version())


def library():
    return _lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return int(t.data_ptr())


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    h = getattr(stream, "cuda_stream", stream)
    return int(h) if h else None


def decode_plan(kv_indptr_host, num_heads: int, num_sms: int = 0):
    """Host plan for a batch.  Returns (plan words as int32 numpy array, workspace bytes)."""
    indptr = np.ascontiguousarray(np.asarray(kv_indptr_host), dtype=np.int32)
    B = indptr.shape[0] - 1
    need = ctypes.c_size_t(0)
    ws = ctypes.c_size_t(0)
    st = _lib.mla_decode_plan(indptr.ctypes.data, B, int(num_heads), int(num_sms), None, 0,
                              ctypes.byref(need), ctypes.byref(ws))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_plan")
    plan = np.zeros(need.value, dtype=np.int32)
    st = _lib.mla_decode_plan(indptr.ctypes.data, B, int(num_heads), int(num_sms), plan.ctypes.data,
                              plan.shape[0], ctypes.byref(need), ctypes.byref(ws))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_plan")
    return plan, int(ws.value)


_H_BATCH, _H_WORKERS, _H_ITEMS = 2, 6, 8      # plan header words (include/mla_decode.h)


def plan_nnz(plan_host) -> int:
    """Token count a plan covers: the largest kv_end of its work items (the
    items tile [0, kv_indptr[batch]) exactly), 0 when it has none."""
    h = np.asarray(plan_host)
    n = int(h[_H_ITEMS])
    if n <= 0:
        return 0
    off = 16 + int(h[_H_WORKERS]) + 1
    return int(h[off + 2: off + 4 * n: 4].max())


def _check_csr(plan_host, kv_indptr, kv_indices, where) -> None:
    """The kernels trust kv_indptr to hold batch + 1 entries and kv_indices
    the slots kv_indptr names (the ABI passes no lengths); with the host plan
    both sizes are checked here, before any launch."""
    h = np.asarray(plan_host)
    batch = int(h[_H_BATCH])
    if kv_indptr is None or kv_indptr.numel() != batch + 1:
        n = 0 if kv_indptr is None else kv_indptr.numel()
        raise ValueError(f"{where}: kv_indptr has {n} entries, the plan was built for {batch + 1}")
    nnz = plan_nnz(h)
    if nnz > 0 and (kv_indices is None or kv_indices.numel() < nnz):
        n = 0 if kv_indices is None else kv_indices.numel()
        raise ValueError(f"{where}: kv_indices has {n} entries, the plan's items reach {nnz}")


def _out_dtype(out, where):
    import torch
    code = {torch.float32: 0, torch.bfloat16: 1}.get(out.dtype)
    if code is None:
        raise MLAError(2, where + ": out dtype")
    return code


def decode_run(plan_host: np.ndarray, plan_dev, q_nope, q_rope, kv_cache, kv_indptr, kv_indices,
               sm_scale: float, out, lse, workspace, stream=None, _entry="mla_decode_run") -> None:
    """Launch the decode (and merge) kernels.  Tensors are torch CUDA tensors:
    q_nope bf16 [B,H,512], q_rope bf16 [B,H,64], kv_cache bf16 [slots,576],
    kv_indptr/kv_indices int32, out fp32 or bf16 [B,H,512], lse fp32 [B,H] or
    None, workspace uint8 (zero-filled before first use)."""
    out_dtype = _out_dtype(out, _entry)
    plan_host = np.ascontiguousarray(plan_host, dtype=np.int32)
    _check_csr(plan_host, kv_indptr, kv_indices, _entry)
    st = getattr(_lib, _entry)(plan_host.ctypes.data, _ptr(plan_dev), _ptr(q_nope), _ptr(q_rope),
                             _ptr(kv_cache), int(kv_cache.shape[0]), _ptr(kv_indptr), _ptr(kv_indices),
                             float(sm_scale), _ptr(out), out_dtype, _ptr(lse), _ptr(workspace),
                             int(workspace.numel() * workspace.element_size()), _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, _entry)


def decode_attend(plan_host, plan_dev, q_nope, q_rope, kv_cache, kv_indptr, kv_indices, sm_scale, out, lse,
                  workspace, stream=None) -> None:
    """The decode kernel alone (whole requests to out/lse, cut ones to partials)."""
    decode_run(plan_host, plan_dev, q_nope, q_rope, kv_cache, kv_indptr, kv_indices, sm_scale, out, lse,
               workspace, stream, _entry="mla_decode_attend")


def decode_merge(plan_host, plan_dev, out, lse, workspace, stream=None) -> None:
    """The plan's LSE merge of partial states (no launch if nothing was cut)."""
    out_dtype = _out_dtype(out, "mla_decode_merge")
    plan_host = np.ascontiguousarray(plan_host, dtype=np.int32)
    st = _lib.mla_decode_merge(plan_host.ctypes.data, _ptr(plan_dev), _ptr(out), out_dtype, _ptr(lse),
                               _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                               _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_merge")


def decode_run_noalloc(plan_host, plan_dev, q_nope, q_rope, kv_cache, kv_indptr, kv_indices, sm_scale, out, lse,
                       stream=None) -> None:
    """mla_decode_run without a workspace: for callers that cannot allocate
    device memory.  Partial states live in the library's static 32 MiB
    device buffer, shared by every call -- calls must not overlap on the GPU."""
    out_dtype = _out_dtype(out, "mla_decode_run_noalloc")
    plan_host = np.ascontiguousarray(plan_host, dtype=np.int32)
    _check_csr(plan_host, kv_indptr, kv_indices, "mla_decode_run_noalloc")
    st = _lib.mla_decode_run_noalloc(plan_host.ctypes.data, _ptr(plan_dev), _ptr(q_nope), _ptr(q_rope),
                                     _ptr(kv_cache), int(kv_cache.shape[0]), _ptr(kv_indptr), _ptr(kv_indices),
                                     float(sm_scale), _ptr(out), out_dtype, _ptr(lse), _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_run_noalloc")


def noalloc_check_errors(stream=None) -> int:
    """Synchronise, read and clear the status word of the static buffer that
    mla_decode_run_noalloc uses on the current device."""
    return int(_lib.mla_noalloc_check_errors(_stream_handle(stream)))


def merge_states(v_partial, s_partial, merge_indptr, out, lse, stream=None) -> None:
    out_dtype = _out_dtype(out, "mla_merge_states")
    B = int(merge_indptr.shape[0]) - 1
    H = int(v_partial.shape[1])
    st = _lib.mla_merge_states(_ptr(v_partial), _ptr(s_partial), _ptr(merge_indptr), B, H, _ptr(out),
                               out_dtype, _ptr(lse), _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_merge_states")


def absorb_query(q_pre, w_kc, q_nope, workspace=None, stream=None) -> None:
    """q_nope[b,h,:] = q_pre[b,h,:] . w_kc[h]: bf16 [B,H,128] x [H,128,512] -> bf16 [B,H,512]."""
    B, H, n = (int(x) for x in q_pre.shape)
    st = _lib.mla_absorb_query(_ptr(q_pre), _ptr(w_kc), _ptr(q_nope), B, H, n, _ptr(workspace),
                               _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_absorb_query")


def project_output(o_lat, w_vc, out, workspace=None, stream=None) -> None:
    """out[b,h,:] = o_lat[b,h,:] . w_vc[h]: bf16 [B,H,512] x [H,512,128] -> fp32 or bf16 [B,H,128]."""
    out_dtype = _out_dtype(out, "mla_project_output")
    B, H = int(o_lat.shape[0]), int(o_lat.shape[1])
    st = _lib.mla_project_output(_ptr(o_lat), _ptr(w_vc), _ptr(out), out_dtype, B, H, int(w_vc.shape[2]),
                                 _ptr(workspace), _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_project_output")


def append_kv(kv_cache, slots, rows, workspace=None, stream=None) -> None:
    """kv_cache[slots[b]] = rows[b]: bf16 [num_slots, 576] <- bf16 [B, 576] at int32 slots [B]."""
    st = _lib.mla_append_kv(_ptr(kv_cache), int(kv_cache.shape[0]), _ptr(slots), _ptr(rows), int(rows.shape[0]),
                            _ptr(workspace), _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_append_kv")


def decode_graph_sizes(max_batch: int, num_heads: int, num_sms: int):
    """(plan_words, workspace_bytes) capacities of mla_decode_run_graph."""
    w, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = _lib.mla_decode_graph_sizes(int(max_batch), int(num_heads), int(num_sms), ctypes.byref(w), ctypes.byref(b))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_graph_sizes")
    return int(w.value), int(b.value)


def decode_run_graph(plan_dev, max_batch, num_heads, num_sms, q_nope, q_rope, kv_cache, kv_indptr, kv_indices,
                     sm_scale, out, lse, workspace, stream=None) -> None:
    """Decode reading its plan only from the device buffer plan_dev (int32, capacity words), so a captured
    graph can be replayed after a new plan (and new CSR arrays) are copied into the same buffers."""
    out_dtype = _out_dtype(out, "mla_decode_run_graph")
    if kv_indptr is None or kv_indptr.numel() != int(max_batch) + 1:
        raise ValueError(f"mla_decode_run_graph: kv_indptr must hold max_batch + 1 = {int(max_batch) + 1} entries")
    st = _lib.mla_decode_run_graph(_ptr(plan_dev), int(plan_dev.numel()), int(max_batch), int(num_heads),
                                   int(num_sms), _ptr(q_nope), _ptr(q_rope), _ptr(kv_cache), int(kv_cache.shape[0]),
                                   _ptr(kv_indptr), _ptr(kv_indices), float(sm_scale), _ptr(out), out_dtype,
                                   _ptr(lse), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                   _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_run_graph")


def decode_fp8_workspace_bytes(plan_host) -> int:
    """Workspace bytes mla_decode_run_fp8 needs for a plan (H 16 or 32)."""
    plan_host = np.ascontiguousarray(plan_host, dtype=np.int32)
    n = ctypes.c_size_t(0)
    st = _lib.mla_decode_fp8_workspace_bytes(plan_host.ctypes.data, ctypes.byref(n))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_fp8_workspace_bytes")
    return int(n.value)


def decode_run_fp8(plan_host, plan_dev, q_nope, q_rope, kv_cache, kv_scale, kv_indptr, kv_indices, sm_scale,
                   out, lse, workspace, stream=None) -> None:
    """Decode over an FP8 cache: kv_cache uint8 [num_slots, 576] E4M3 codes (value = code x kv_scale);
    other tensors as for decode_run; workspace of decode_fp8_workspace_bytes(plan) bytes, zero-filled once."""
    out_dtype = _out_dtype(out, "mla_decode_run_fp8")
    plan_host = np.ascontiguousarray(plan_host, dtype=np.int32)
    _check_csr(plan_host, kv_indptr, kv_indices, "mla_decode_run_fp8")
    st = _lib.mla_decode_run_fp8(plan_host.ctypes.data, _ptr(plan_dev), _ptr(q_nope), _ptr(q_rope), _ptr(kv_cache),
                                 int(kv_cache.shape[0]), float(kv_scale), _ptr(kv_indptr), _ptr(kv_indices),
                                 float(sm_scale), _ptr(out), out_dtype, _ptr(lse), _ptr(workspace),
                                 int(workspace.numel() * workspace.element_size()), _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_run_fp8")


def append_kv_fp8(kv_cache, slots, rows, kv_scale, workspace=None, stream=None) -> None:
    """kv_cache[slots[b]] = E4M3(rows[b] / kv_scale): uint8 [num_slots, 576] <- bf16 [B, 576]."""
    st = _lib.mla_append_kv_fp8(_ptr(kv_cache), int(kv_cache.shape[0]), _ptr(slots), _ptr(rows), int(rows.shape[0]),
                                float(kv_scale), _ptr(workspace), _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_append_kv_fp8")


def decode_run_multi_query(plan_host, plan_dev, q_len, q_nope, q_rope, kv_cache, kv_indptr, kv_indices, sm_scale,
                           out, lse, workspace, stream=None) -> None:
    """q_len draft tokens per request in one pass: q [B, q_len, H, 576 split], out [B, q_len, H, 512]."""
    out_dtype = _out_dtype(out, "mla_decode_run_multi_query")
    plan_host = np.ascontiguousarray(plan_host, dtype=np.int32)
    _check_csr(plan_host, kv_indptr, kv_indices, "mla_decode_run_multi_query")
    st = _lib.mla_decode_run_multi_query(plan_host.ctypes.data, _ptr(plan_dev), int(q_len), _ptr(q_nope),
                                         _ptr(q_rope), _ptr(kv_cache), int(kv_cache.shape[0]), _ptr(kv_indptr),
                                         _ptr(kv_indices), float(sm_scale), _ptr(out), out_dtype, _ptr(lse),
                                         _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                         _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_run_multi_query")


def decode_run_tree(plan_host, plan_dev, parents, tree_masks, q_nope, q_rope, kv_cache, kv_indptr, kv_indices,
                    sm_scale, out, lse, workspace, stream=None) -> None:
    """A tree of W draft tokens per request in one pass: parents device int32 [B, W] (each draft's parent, an
    earlier draft, or -1), tree_masks device int64 [B, W] scratch; q [B, W, H, 576 split], out [B, W, H, 512]."""
    out_dtype = _out_dtype(out, "mla_decode_run_tree")
    plan_host = np.ascontiguousarray(plan_host, dtype=np.int32)
    _check_csr(plan_host, kv_indptr, kv_indices, "mla_decode_run_tree")
    W = int(parents.shape[-1])
    if tree_masks.numel() < parents.numel() or tree_masks.element_size() != 8:
        raise MLAError(1, "mla_decode_run_tree: tree_masks must hold one 8-byte word per draft")
    st = _lib.mla_decode_run_tree(plan_host.ctypes.data, _ptr(plan_dev), W, _ptr(parents), _ptr(tree_masks),
                                  _ptr(q_nope), _ptr(q_rope), _ptr(kv_cache), int(kv_cache.shape[0]),
                                  _ptr(kv_indptr), _ptr(kv_indices), float(sm_scale), _ptr(out), out_dtype,
                                  _ptr(lse), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                  _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_run_tree")


def merge_two_states(o_a, lse_a, o_b, lse_b, out, lse, stream=None) -> None:
    """Row-wise LSE merge of two fp32 states [..., 512] / [...] into out (fp32 or bf16) and lse."""
    out_dtype = _out_dtype(out, "mla_merge_two_states")
    rows = int(lse_a.numel())
    st = _lib.mla_merge_two_states(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), rows, _ptr(out), out_dtype,
                                   _ptr(lse), _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_merge_two_states")


def step_staging_bytes(batch: int, num_heads: int, nnz: int, plan_words: int, out_dtype: int) -> int:
    return int(_lib.mla_step_staging_bytes(batch, num_heads, nnz, plan_words, out_dtype))


def decode_step_host(q_nope, q_rope, kv_indptr, kv_indices, kv_cache, sm_scale, out, lse, plan, staging, workspace,
                     stream=None, copy_in_stream=None, copy_out_stream=None) -> None:
    """One step from host tensors (pinned for asynchronous copies): plan, copy in, run, copy out on `stream`.
    `plan` is a host int32 tensor with room for the plan words."""
    out_dtype = _out_dtype(out, "mla_decode_step_host")
    B, H = int(q_nope.shape[0]), int(q_nope.shape[1])
    if kv_indptr.numel() != B + 1 or kv_indices.numel() < int(kv_indptr[-1]):
        raise ValueError("mla_decode_step_host: kv_indptr must hold batch + 1 entries and kv_indices the "
                         "kv_indptr[batch] slots it names")
    st = _lib.mla_decode_step_host(_ptr(q_nope), _ptr(q_rope), _ptr(kv_indptr), _ptr(kv_indices), B, H,
                                   _ptr(kv_cache), int(kv_cache.shape[0]), float(sm_scale), _ptr(out), out_dtype,
                                   _ptr(lse), _ptr(plan), int(plan.numel()), _ptr(staging), int(staging.numel()),
                                   _ptr(workspace), int(workspace.numel()), _stream_handle(stream),
                                   None if copy_in_stream is None else _stream_handle(copy_in_stream),
                                   None if copy_out_stream is None else _stream_handle(copy_out_stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_decode_step_host")


def check_errors(workspace, stream=None) -> int:
    """Synchronise, read and clear the device status; returns the status code."""
    return int(_lib.mla_check_errors(_ptr(workspace), _stream_handle(stream)))


def probe_wait_limit(workspace, stream=None) -> None:
    """Launch the bounded-wait diagnostic: a wait that nothing completes gives up
    after the kernels' wait limit and leaves MLA_ERR_TIMEOUT in the status word."""
    st = _lib.mla_probe_wait_limit(_ptr(workspace), _stream_handle(stream))
    if st != MLA_OK:
        raise MLAError(st, "mla_probe_wait_limit")


class Decoder:
    """Convenience holder: plan once per batch shape, then run on device tensors."""

    def __init__(self, kv_indptr_host, num_heads: int, device="cuda", num_sms: int = 0):
        import torch
        self.plan_host, self.workspace_bytes = decode_plan(kv_indptr_host, num_heads, num_sms)
        self.plan_dev = torch.from_numpy(self.plan_host).to(device)
        self.workspace = torch.zeros(max(self.workspace_bytes, 256), dtype=torch.uint8, device=device)
        self.num_heads = num_heads
        self.batch = int(np.asarray(kv_indptr_host).shape[0]) - 1
        self.nnz = int(np.asarray(kv_indptr_host)[-1])

    @property
    def header(self):
        return self.plan_host[:16]

    def run(self, q_nope, q_rope, kv_cache, kv_indptr, kv_indices, sm_scale, out, lse, stream=None):
        decode_run(self.plan_host, self.plan_dev, q_nope, q_rope, kv_cache, kv_indptr, kv_indices,
                   sm_scale, out, lse, self.workspace, stream)

    def attend(self, q_nope, q_rope, kv_cache, kv_indptr, kv_indices, sm_scale, out, lse, stream=None):
        decode_attend(self.plan_host, self.plan_dev, q_nope, q_rope, kv_cache, kv_indptr, kv_indices,
                      sm_scale, out, lse, self.workspace, stream)

    def merge(self, out, lse, stream=None):
        decode_merge(self.plan_host, self.plan_dev, out, lse, self.workspace, stream)

    @property
    def has_merge(self) -> bool:
        return int(self.plan_host[10]) > 0

    def check(self, stream=None) -> int:
        return check_errors(self.workspace, stream)
