#!/usr/bin/env python
"""Benchmark of absorbed MLA decode on GB300 (one JSON line on stdout).

A step is one whole decode pass (mla_decode_attend + mla_decode_merge) over one
synthetic batch whose inputs are already resident in HBM.  Default workload:
the ragged serving batch (B=256, H=128, contexts lognormal around 1500 clipped
to [16, 32768], page size 1, 2^20-slot pool); ``--workload 1..5`` picks another.
The other >= 4k-context workloads of the family (V2-Lite B=64/H=16, V3
B=128/H=128 at 4096, long B=2/H=128 at 64k + 128k) are measured in the same
run under ``per_config`` (step and decode kernel alone, each one CUDA-graph
replay over rotating input sets), with their side legs.

Timing: W untimed warm-up steps, then exactly K steps run back to back (as a
decode loop runs them) between two CUDA events on the launching stream,
bracketed by a barrier and torch.cuda.synchronize() on both sides; the max
over ranks is reported.  L2 cannot help: step k reads input set k mod R, and
the R sets (each with its own KV pool, query, indices) are chosen so that the
cache bytes the other R-1 steps stream in between exceed 4x the L2 size.
The decode kernel's own time (the roofline's "achieved") is taken in a second
pass: K decode launches alone (no merge) over the same rotation, captured as
one CUDA graph and timed as one replay; a third pass reports the step with a
256 MiB L2-flushing write (outside the events) before each step.
``--gpus N`` under torchrun runs N independent replicas (the path needs no
collective).  ``--impl reference`` times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MLA decode µs/step and latent-KV GB/s as % of GB300 HBM roofline (1 GPU)"
UNIT = "us/step"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def algorithmic_work(batch):
    """Bytes and flops the path must move / compute for one step (not the
    decompressed work absorption avoids): every cache row once, the indices,
    q, the fp32 output and lse; flops 2*576 (QK) + 2*512 (PV) per head-token."""
    B, H, nnz = batch.batch, batch.heads, batch.nnz
    bytes_ = nnz * 1152 + nnz * 4 + B * H * 576 * 2 + B * H * 512 * 4 + B * H * 4 + (B + 1) * 4
    flops = nnz * H * 2 * (576 + 512)
    return bytes_, flops


KERNEL_SOURCES = {
    "swab": ("mla_swab.cu", "mla_device.cuh", "mla_internal.h", "mla_launch.h"),
    "pair": ("mla_pair.cu", "mla_device.cuh", "mla_internal.h", "mla_launch.h"),
}


_C_TOKENS = re.compile(r'"(?:\\.|[^"\\\n])*"|//[^\n]*|/\*.*?\*/', re.S)


def _code_only(text):
    """C/CUDA source with its comments removed (string literals kept),
    trailing blanks and empty lines dropped."""
    text = _C_TOKENS.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def host_plan_us(binding, kv_indptr, heads, words, num_sms=0, repeats=20):
    """Median time of one mla_decode_plan call into a preallocated buffer
    (the call mla_decode_step_host makes every step), in microseconds."""
    import ctypes

    import numpy as np
    lib = binding.library()
    ind = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    plan = np.empty(words, dtype=np.int32)
    need, ws = ctypes.c_size_t(0), ctypes.c_size_t(0)
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        st = lib.mla_decode_plan(ind.ctypes.data, ind.size - 1, heads, num_sms, plan.ctypes.data, words,
                                 ctypes.byref(need), ctypes.byref(ws))
        times.append((time.perf_counter() - t0) * 1e6)
        if st != 0:
            raise RuntimeError(f"mla_decode_plan returned {st}")
    return statistics.median(times)


def kernel_source_sha(kernel):
    """Digest of the code (not the comments) of the sources that make up one
    decode kernel."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_latent_kv_absorbed_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload_name, kernel):
    """DRAM bytes (read + write) per decode-kernel launch from the committed
    ncu summary profiles/ncu_traffic.txt, or None when there is no entry or
    the entry was taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) == 4 and not line.startswith("#") and parts[0] == workload_name \
                        and parts[1] == kernel:
                    return float(parts[2]) if parts[3] == kernel_source_sha(kernel) else None
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def max_over_ranks(value, pg, device=None):
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def cpu_oracle_sample(batch, budget_s):
    """Time the fp64 oracle on the first requests of the batch until about
    budget_s of CPU work, and scale to the whole batch by tokens."""
    from oracle import mla_oracle as O
    reqs, t_total, tok = [], 0.0, 0
    order = list(range(batch.batch))
    for b in order:
        t0 = time.perf_counter()
        O.decode_attention(batch.q_nope, batch.q_rope, batch.kv_cache, batch.kv_indptr, batch.kv_indices,
                           batch.sm_scale, requests=[b])
        t_total += time.perf_counter() - t0
        reqs.append(b)
        tok += int(batch.kv_indptr[b + 1] - batch.kv_indptr[b])
        if t_total >= budget_s:
            break
    scale = batch.nnz / max(tok, 1)
    return t_total * scale * 1e6, len(reqs), tok


def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def run_reference(args, batch, rank, pg):
    """--impl reference: the fp64 oracle on the host cores, bounded sample per step."""
    if pg is not None and rank != 0:
        return 0
    per_step_budget = max(0.5, args.reference_budget_s / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_oracle_sample(batch, per_step_budget)
    vals, samples = [], None
    for _ in range(args.steps):
        us, nreq, tok = cpu_oracle_sample(batch, per_step_budget)
        vals.append(us)
        samples = (nreq, tok)
    value = statistics.mean(vals)
    cores = oracle_threads()
    sample = f"first {samples[0]} requests ({samples[1]} of {batch.nnz} tokens) per step, scaled by tokens"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(batch, args, host=True),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(batch, args, rotate=None, host=False):
    spec = batch.spec
    if host:
        l2 = ("not applicable: the fp64 oracle runs on the host CPU from host memory (numpy); no GPU cache "
              "is involved")
    elif rotate and rotate[0] > 1:
        l2 = ("inputs larger than L2: step k reads input set k mod %d (own KV pool, q, indices), "
              "the other sets stream %.0f MB of cache in between" % rotate)
    elif rotate:
        l2 = "one input set, steps back to back (profiling run; not a benchmark number)"
    else:
        l2 = "flushed before every timed step (256 MiB write, outside the events)"
    return {"workload": spec.name if spec else "custom", "batch": batch.batch, "heads": batch.heads,
            "kv_lora_rank": 512, "qk_rope_head_dim": 64, "nnz": batch.nnz, "pool_slots": batch.pool,
            "max_context": int(batch.lengths.max()), "page_size": 1, "out_dtype": "fp32",
            "l2": l2, "parallelism": f"replicas x{args.gpus}"}


def time_head_products(batch, dev, peaks):
    """The two per-head products around the decode at this workload's B and H
    (query absorption q.w_kc, output projection o_lat.w_vc), each timed over
    back-to-back launches that rotate through input sets totalling more than
    4x L2, against its own roofline.  Not part of the decode step."""
    import numpy as np
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads
    Bn, H = batch.batch, batch.heads
    x = workloads.make_head_product_inputs(Bn, H, seed=workloads.SEED_BASE + 900)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    q_pre, w_kc, w_vc = bf(x.q_pre), bf(x.w_kc), bf(x.w_vc)
    o_lat = torch.randn((Bn, H, 512), device=dev).to(torch.bfloat16)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    res = {}
    for name in ("absorb", "project"):
        if name == "absorb":
            a, w = q_pre, w_kc
            out_shape, out_dt, out_size = (Bn, H, 512), torch.bfloat16, 2
            K, N = 128, 512
        else:
            a, w = o_lat, w_vc
            out_shape, out_dt, out_size = (Bn, H, 128), torch.float32, 4
            K, N = 512, 128
        bytes_alg = H * K * N * 2 + Bn * H * K * 2 + Bn * H * N * out_size
        flops = 2 * Bn * H * K * N
        R = max(20, math.ceil(4 * l2 / bytes_alg) + 1)
        sets = [(a.clone(), w.clone(), torch.empty(out_shape, dtype=out_dt, device=dev)) for _ in range(R)]
        fn = binding.absorb_query if name == "absorb" else binding.project_output
        for k in range(3):
            fn(*sets[k % R])
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for k in range(R):
            fn(*sets[k])
        e1.record()
        torch.cuda.synchronize()
        us_eager = e0.elapsed_time(e1) * 1e3 / R
        # the same launches captured in a CUDA graph: the device time without
        # the host's per-call work (argument checks, tensor-map encoding)
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for k in range(R):
                    fn(*sets[k], stream=cap)
        torch.cuda.current_stream().wait_stream(cap)
        g.replay()
        torch.cuda.synchronize()
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / R
        t_hbm = bytes_alg / (peaks["hbm_gbs"] * 1e9) * 1e6
        t_tc = flops / (peaks["bf16_tflops"] * 1e12) * 1e6
        res[name] = {"us": us, "us_eager": us_eager, "roofline_us": max(t_hbm, t_tc), "frac": max(t_hbm, t_tc) / us,
                     "bound": "hbm" if t_hbm >= t_tc else "tensor", "algorithmic_bytes": bytes_alg,
                     "algorithmic_flops": flops, "launches": R}
        del sets
    res["note"] = ("q_pre [B,H,128] . w_kc [H,128,512] -> bf16, o_lat [B,H,512] . w_vc [H,512,128] -> fp32; "
                   "synthetic weights N(0,1/fan_in); launches rotating input sets > 4x L2, timed as one CUDA-graph replay "
                   "(us) and as eager back-to-back calls (us_eager)")
    return res


def time_multi_query(batch, dev, peaks, kv, indptr_d, indices_d):
    """Draft verification at this workload's lengths, at two draft counts:
    q_len = 64 / H (the q_len x H = 64 rows run on the two-CTA kernel) and
    q_len = 32 / H (32 rows: the few-heads kernel), each timed over
    back-to-back launches that rotate KV copies larger than 4x L2.  Only for
    H <= 32 (at H = 128 the rows would exceed 128)."""
    import numpy as np
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    Bn, H = batch.batch, batch.heads
    if H > 32:
        return None
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, math.ceil(4 * l2 / (batch.nnz * 1152)) + 1)
    kvs = [kv] + [kv.clone() for _ in range(R - 1)]

    def one(q_len):
        qn = torch.randn((Bn, q_len, H, 512), device=dev).to(torch.bfloat16)
        qr = torch.randn((Bn, q_len, H, 64), device=dev).to(torch.bfloat16)
        plan, ws_bytes = binding.decode_plan(batch.kv_indptr, q_len * H)
        plan_d = torch.from_numpy(plan).to(dev)
        ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        out = torch.empty((Bn, q_len, H, 512), dtype=torch.float32, device=dev)
        lse = torch.empty((Bn, q_len, H), dtype=torch.float32, device=dev)
        run = lambda k: binding.decode_run_multi_query(plan, plan_d, q_len, qn, qr, kvs[k % R], indptr_d, indices_d,
                                                       batch.sm_scale, out, lse, ws)
        for k in range(3):
            run(k)
        torch.cuda.synchronize()
        n = max(20, R)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for k in range(n):
            run(k)
        e1.record()
        torch.cuda.synchronize()
        st = binding.check_errors(ws)
        if st != 0:
            raise RuntimeError(f"device status after multi-query: {binding.status_string(st)}")
        us = e0.elapsed_time(e1) * 1e3 / n
        rows = Bn * q_len * H
        bytes_alg = batch.nnz * 1152 + batch.nnz * 4 + rows * (576 * 2 + 512 * 4 + 4) + (Bn + 1) * 4
        flops = 2176 * H * sum(max(0, int(L) - q_len + 1 + i) for L in batch.lengths for i in range(q_len))
        t = max(bytes_alg / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12)) * 1e6
        return q_len, us, t

    q_len, us, t = one(64 // H)
    res = {"q_len": q_len, "heads_per_query": H, "us": us, "roofline_us": t, "frac": t / us}
    if 32 // H >= 2:
        q2, us2, t2 = one(32 // H)
        res["q_len_32_rows"] = {"q_len": q2, "us": us2, "roofline_us": t2, "frac": t2 / us2,
                                "kernel": "few-heads (32 rows)"}
    res["note"] = ("q_len draft tokens per request verified in one pass (mla_decode_run_multi_query); the main "
                   "figure is 64 rows (two-CTA kernel), q_len_32_rows the few-heads kernel; synthetic queries, this "
                   "workload's contexts; back-to-back launches over KV copies > 4x L2")
    del kvs
    return res


def topk_tree_parents(width, topk=2):
    """Parent array of a draft tree grown breadth first, every draft getting
    `topk` children until `width` drafts exist (-1: a child of the verified
    context).  topk = 2, width = 8: [-1, 0, 0, 1, 1, 2, 2, 3], depth 4."""
    par = [-1]
    node = 0
    while len(par) < width:
        for _ in range(topk):
            if len(par) < width:
                par.append(node)
        node += 1
    return par


def time_tree(batch, dev, peaks, kv, indptr_d, indices_d):
    """Tree-shaped draft verification (mla_decode_run_tree) at this
    workload's contexts: a top-2 tree of W = 128 // H drafts per request
    (every query sees the context and its ancestors), and for comparison the
    chain of W drafts (mla_decode_run_multi_query), each over back-to-back
    launches that rotate KV copies larger than 4x L2.  Only for H <= 32."""
    import numpy as np
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    Bn, H = batch.batch, batch.heads
    if H > 32:
        return None
    W = 128 // H
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, math.ceil(4 * l2 / (batch.nnz * 1152)) + 1)
    kvs = [kv] + [kv.clone() for _ in range(R - 1)]
    par_host = np.tile(np.array(topk_tree_parents(W), dtype=np.int32), (Bn, 1))
    parents = torch.from_numpy(par_host).to(dev)
    masks = torch.zeros((Bn, W), dtype=torch.int64, device=dev)
    qn = torch.randn((Bn, W, H, 512), device=dev).to(torch.bfloat16)
    qr = torch.randn((Bn, W, H, 64), device=dev).to(torch.bfloat16)
    plan, ws_bytes = binding.decode_plan(batch.kv_indptr, W * H)
    plan_d = torch.from_numpy(plan).to(dev)
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    out = torch.empty((Bn, W, H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((Bn, W, H), dtype=torch.float32, device=dev)
    runs = {
        "tree": lambda k: binding.decode_run_tree(plan, plan_d, parents, masks, qn, qr, kvs[k % R], indptr_d,
                                                  indices_d, batch.sm_scale, out, lse, ws),
        "chain": lambda k: binding.decode_run_multi_query(plan, plan_d, W, qn, qr, kvs[k % R], indptr_d, indices_d,
                                                          batch.sm_scale, out, lse, ws),
    }
    res = {"drafts": W, "topk": 2, "parents": topk_tree_parents(W), "heads_per_query": H}
    anc = []
    for i, p_ in enumerate(res["parents"]):
        anc.append(1 if p_ < 0 else anc[p_] + 1)          # drafts each query sees (its depth)
    for name, run in runs.items():
        for k in range(3):
            run(k)
        torch.cuda.synchronize()
        n = max(20, R)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for k in range(n):
            run(k)
        e1.record()
        torch.cuda.synchronize()
        st = binding.check_errors(ws)
        if st != 0:
            raise RuntimeError(f"device status after the {name} verification: {binding.status_string(st)}")
        us = e0.elapsed_time(e1) * 1e3 / n
        rows = Bn * W * H
        bytes_alg = batch.nnz * 1152 + batch.nnz * 4 + rows * (576 * 2 + 512 * 4 + 4) + (Bn + 1) * 4
        seen = anc if name == "tree" else [i + 1 for i in range(W)]
        flops = 2176 * H * sum(max(0, int(L) - W) + d for L in batch.lengths for d in seen)
        t = max(bytes_alg / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12)) * 1e6
        res[name] = {"us": us, "roofline_us": t, "frac": t / us}
    res["note"] = ("W draft tokens per request verified in one pass over this workload's contexts; tree: a top-2 "
                   "breadth-first tree (parents as listed), each query seeing the context and its ancestors "
                   "(ancestor masks built by a small kernel every call); chain: the same W drafts in a line; "
                   "synthetic queries; back-to-back launches over KV copies > 4x L2")
    del kvs
    return res


def cascade_csr(batch):
    """Host CSR arrays of the shared-prefix leg (H <= 32): a prefix of
    min(4096, pool) distinct slots; G pseudo-requests of 128 // H requests'
    rows over it (p_ptr, p_ind); the workload's contexts as suffixes, padded
    with empty requests to whole groups (s_ptr); and each request over prefix
    + suffix (f_ptr, f_ind).  Raises unless every index array holds exactly
    the slots its kv_indptr names."""
    import numpy as np
    Bn, H = batch.batch, batch.heads
    Lp, group = min(4096, batch.pool), 128 // H            # distinct prefix slots: at most the pool
    G = (Bn + group - 1) // group
    Bp = G * group                                           # padded to whole groups
    prefix = np.random.default_rng(11).permutation(batch.pool)[:Lp].astype(np.int32)
    p_ptr = np.arange(G + 1, dtype=np.int32) * Lp
    p_ind = np.tile(prefix, G)
    s_ptr = np.concatenate([batch.kv_indptr, np.full(Bp - Bn, batch.kv_indptr[-1])]).astype(np.int32)
    f_ptr = (s_ptr + np.arange(Bp + 1, dtype=np.int32) * Lp).astype(np.int32)
    f_ind = np.concatenate([np.concatenate([prefix, batch.kv_indices[s_ptr[b]:s_ptr[b + 1]]]) for b in range(Bp)])
    if not (len(prefix) == Lp and len(p_ind) == p_ptr[-1] and len(batch.kv_indices) == s_ptr[-1] == batch.nnz
            and len(f_ind) == f_ptr[-1]):
        raise RuntimeError("cascade index arrays do not match their kv_indptr")
    return {"prefix_rows": Lp, "group": group, "groups": G, "padded_batch": Bp, "p_ptr": p_ptr, "p_ind": p_ind,
            "s_ptr": s_ptr, "f_ptr": f_ptr, "f_ind": f_ind}


def time_cascade(batch, dev, peaks):
    """Shared-prefix cascade at this workload's shape: every request gets a
    shared prefix of min(4096, pool) rows in front of its own context (the workload's rows
    as suffix).  Cascade = prefix pass (the query rows of 128 // H requests as
    the heads of one pseudo-request, so the prefix is read once per group),
    suffix pass, two-state merge; flat = one decode over prefix + suffix rows
    per request.  Each captured in a CUDA graph and replayed back to back.
    Only for H <= 32."""
    import numpy as np
    import torch
    from mla_latent_kv_absorbed_gb300 import binding
    Bn, H = batch.batch, batch.heads
    if H > 32:
        return None
    c = cascade_csr(batch)
    Lp, group, G, Bp = c["prefix_rows"], c["group"], c["groups"], c["padded_batch"]
    p_ptr, s_ptr, f_ptr, f_ind = c["p_ptr"], c["s_ptr"], c["f_ptr"], c["f_ind"]
    ti = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    kv = torch.from_numpy(np.ascontiguousarray(batch.kv_cache).view(np.int16)).view(torch.bfloat16).to(dev)
    qn = torch.randn((Bp, H, 512), device=dev).to(torch.bfloat16)
    qr = torch.randn((Bp, H, 64), device=dev).to(torch.bfloat16)
    sc = batch.sm_scale
    # prefix pass: G pseudo-requests of group x H rows over the same prefix rows
    dec_p = binding.Decoder(p_ptr, group * H, device=dev)
    p_ind = ti(c["p_ind"])
    o_p = torch.empty((Bp, H, 512), dtype=torch.float32, device=dev)
    l_p = torch.empty((Bp, H), dtype=torch.float32, device=dev)
    # suffix pass: the workload's contexts (padding requests empty)
    dec_s = binding.Decoder(s_ptr, H, device=dev)
    s_ind = ti(batch.kv_indices)
    o_s, l_s = torch.empty_like(o_p), torch.empty_like(l_p)
    out, lse = torch.empty_like(o_p), torch.empty_like(l_p)
    # flat: each request over prefix + suffix
    dec_f = binding.Decoder(f_ptr, H, device=dev)
    f_ind_d = ti(f_ind)
    o_f, l_f = torch.empty_like(o_p), torch.empty_like(l_p)
    p_ptr_d, s_ptr_d, f_ptr_d = ti(p_ptr), ti(s_ptr), ti(f_ptr)

    def cascade(stream=None):
        dec_p.run(qn.view(G, group * H, 512), qr.view(G, group * H, 64), kv, p_ptr_d, p_ind, sc, o_p, l_p,
                  stream=stream)
        dec_s.run(qn, qr, kv, s_ptr_d, s_ind, sc, o_s, l_s, stream=stream)
        binding.merge_two_states(o_p, l_p, o_s, l_s, out, lse, stream=stream)

    def flat(stream=None):
        dec_f.run(qn, qr, kv, f_ptr_d, f_ind_d, sc, o_f, l_f, stream=stream)

    # each variant captured once in a CUDA graph (no host work between its
    # launches), replayed back to back
    res = {}
    cap = torch.cuda.Stream(device=dev)
    for name, fn in (("cascade", cascade), ("flat", flat)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                fn(stream=cap)
        torch.cuda.current_stream().wait_stream(cap)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        n = 20
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        res[name + "_us"] = e0.elapsed_time(e1) * 1e3 / n
        del g
    for d in (dec_p, dec_s, dec_f):
        if d.check() != 0:
            raise RuntimeError("device status after cascade")
    diff = (out - o_f).abs().max().item()
    res.update({"prefix_rows": Lp, "requests": Bn, "requests_per_prefix_pass": group,
                "max_abs_diff_cascade_vs_flat": diff,
                "note": f"shared prefix of {Lp} rows in front of each context; cascade = prefix pass with the query "
                        "rows of 128 // H requests as one pseudo-request's heads + suffix pass + mla_merge_two_states; "
                        "CUDA-graph replays; L2 not flushed (the prefix rows are reused by design)"})
    return res


def time_fp8(batch, dev, peaks, step_us_bf16, indptr_d, indices_d):
    """The same decode over an FP8 (E4M3) copy of the cache (mla_decode_run_fp8:
    at H <= 32 a query-prep kernel, the few-heads FP8 decode and the merge; at
    H >= 48 the two-CTA FP8 decode and the merge).  Synthetic codes with kv_scale
    2^-5; R pool copies whose touched bytes exceed 4x L2 are rotated inside one
    captured CUDA graph, replayed after warm-up.  Flops as for bf16 (the
    roofline takes the larger of the byte and flop times)."""
    import numpy as np
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads as W
    Bn, H = batch.batch, batch.heads
    spec_seed = 20261200 + 80 + (batch.spec.number if batch.spec else 0)
    codes = torch.from_numpy(W.make_fp8_cache(batch.pool, spec_seed)).to(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, math.ceil(4 * l2 / (batch.nnz * 576)) + 1)
    kvs = [codes] + [codes.clone() for _ in range(R - 1)]
    plan, _ = binding.decode_plan(batch.kv_indptr, H)
    plan_d = torch.from_numpy(plan).to(dev)
    ws = torch.zeros(binding.decode_fp8_workspace_bytes(plan), dtype=torch.uint8, device=dev)
    qn = torch.from_numpy(np.ascontiguousarray(batch.q_nope).view(np.int16)).view(torch.bfloat16).to(dev)
    qr = torch.from_numpy(np.ascontiguousarray(batch.q_rope).view(np.int16)).view(torch.bfloat16).to(dev)
    out = torch.empty((Bn, H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((Bn, H), dtype=torch.float32, device=dev)
    run = lambda k, stream=None: binding.decode_run_fp8(plan, plan_d, qn, qr, kvs[k % R], W.FP8_KV_SCALE, indptr_d,
                                                         indices_d, batch.sm_scale, out, lse, ws, stream=stream)
    for k in range(3):
        run(k)
    torch.cuda.synchronize()
    st = binding.check_errors(ws)
    if st != 0:
        raise RuntimeError(f"device status after the FP8 decode: {binding.status_string(st)}")
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            for k in range(R):
                run(k, stream=cap)
    torch.cuda.current_stream().wait_stream(cap)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    reps = max(3, math.ceil(60 / R))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    st = binding.check_errors(ws)
    if st != 0:
        raise RuntimeError(f"device status after the FP8 decode: {binding.status_string(st)}")
    us = e0.elapsed_time(e1) * 1e3 / (reps * R)
    bytes_alg = batch.nnz * 576 + batch.nnz * 4 + Bn * H * (576 * 2 + 512 * 4 + 4) + (Bn + 1) * 4
    flops = batch.nnz * H * 2176
    t = max(bytes_alg / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 2e12)) * 1e6
    del kvs, g
    return {"us": us, "roofline_us": t, "frac": t / us, "algorithmic_bytes": bytes_alg,
            "bound": "hbm" if bytes_alg / (peaks["hbm_gbs"] * 1e9) >= flops / (peaks["bf16_tflops"] * 2e12) else "tensor",
            "fp8_peak_note": "fp8 dense tensor peak taken as 2x the measured bf16 peak (the nominal ratio)",
            "latent_kv_gbs": batch.nnz * 576 / (us * 1e-6) / 1e9, "speedup_vs_bf16_step": step_us_bf16 / us,
            "kv_scale": W.FP8_KV_SCALE,
            "note": "FP8 (E4M3) cache, one byte per value; decode (tcgen05 kind::f8f6f4; H <= 32 after a query-prep "
                    "kernel, H >= 48 the two-CTA kernel) + merge per step; synthetic codes; R KV copies > 4x L2 "
                    "rotated inside one CUDA graph"}


def graph_ms_per_call(fn, n, stream, dev):
    """Capture n calls fn(k, stream) as one CUDA graph, replay it once
    untimed, then time one replay with events on `stream`: milliseconds per
    call."""
    import torch
    cap = torch.cuda.Stream(dev)
    g = torch.cuda.CUDAGraph()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            for k in range(n):
                fn(k, cap)
    stream.wait_stream(cap)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) / n


class DecodeInputs:
    """One workload on the device: R input sets (KV pool, q, indices) such
    that the other R-1 steps of a back-to-back run stream more than 4x L2 of
    cache rows, the decoder (plan + workspace) and the outputs."""

    def __init__(self, batch, dev, args):
        import numpy as np
        import torch
        from mla_latent_kv_absorbed_gb300 import binding
        self.batch, self.dev = batch, dev
        bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        q_nope, q_rope, self.kv = bf(batch.q_nope), bf(batch.q_rope), bf(batch.kv_cache)
        self.indptr_d = torch.from_numpy(batch.kv_indptr).to(dev)
        self.indices_d = torch.from_numpy(batch.kv_indices).to(dev)
        Bn, H = batch.batch, batch.heads
        self.out = torch.empty((Bn, H, 512), dtype=torch.float32, device=dev)
        self.lse = torch.empty((Bn, H), dtype=torch.float32, device=dev)
        self.dec = binding.Decoder(batch.kv_indptr, H, device=dev)
        l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
        self.step_kv_bytes = batch.nnz * 1152
        self.R = args.sets if args.sets > 0 else max(2, math.ceil(4 * l2_bytes / self.step_kv_bytes) + 1)
        self.sets = [(q_nope, q_rope, self.kv, self.indices_d)]
        for _ in range(self.R - 1):
            self.sets.append((q_nope.clone(), q_rope.clone(), self.kv.clone(), self.indices_d.clone()))

    def attend(self, k, st):
        qn, qr, kvc, ind = self.sets[k % self.R]
        self.dec.attend(qn, qr, kvc, self.indptr_d, ind, self.batch.sm_scale, self.out, self.lse, st)

    def step(self, k, st):
        self.attend(k, st)
        self.dec.merge(self.out, self.lse, st)

    def check(self, stream, where):
        from mla_latent_kv_absorbed_gb300 import binding
        st = self.dec.check(stream)
        if st != 0:
            raise RuntimeError(f"device status {where}: {binding.status_string(st)}")

    @property
    def rotate(self):
        return (self.R, (self.R - 1) * self.step_kv_bytes / 1e6)


def time_absorbing_step(x, dev, args, peaks, decode_step_ms):
    """A whole absorbing decode step at this workload's shape, timed as one
    CUDA-graph replay of K steps over the rotating input sets: query
    absorption (q_pre . w_kc -> the decode's q_nope), the append of one new
    cache row per request (its context's last slot), the decode and merge
    (bf16 output) and the output projection (o_lat . w_vc -> fp32).  Every
    launch is a programmatic dependent of the one before it, so each kernel's
    setup overlaps its predecessor's tail."""
    import numpy as np
    import torch
    from mla_latent_kv_absorbed_gb300 import binding, workloads
    b = x.batch
    Bn, H = b.batch, b.heads
    stream = torch.cuda.current_stream(dev)
    hp = workloads.make_head_product_inputs(Bn, H, seed=workloads.SEED_BASE + 901)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    q_pre, w_kc, w_vc = bf(hp.q_pre), bf(hp.w_kc), bf(hp.w_vc)
    lengths = np.diff(b.kv_indptr)
    if (lengths < 1).any():
        return None
    slots = torch.from_numpy(b.kv_indices[b.kv_indptr[1:] - 1].astype(np.int32)).to(dev)
    new_rows = torch.randn((Bn, 576), device=dev).to(torch.bfloat16)
    o_lat = torch.empty((Bn, H, 512), dtype=torch.bfloat16, device=dev)
    out = torch.empty((Bn, H, 128), dtype=torch.float32, device=dev)

    def step(k, st):
        qn, qr, kvc, ind = x.sets[k % x.R]
        binding.absorb_query(q_pre, w_kc, qn, stream=st)
        binding.append_kv(kvc, slots, new_rows, stream=st)
        x.dec.attend(qn, qr, kvc, x.indptr_d, ind, b.sm_scale, o_lat, x.lse, st)
        x.dec.merge(o_lat, x.lse, st)
        binding.project_output(o_lat, w_vc, out, stream=st)

    for k in range(max(3, x.R)):
        step(k, stream)
    x.check(stream, "after the absorbing step")
    ms = graph_ms_per_call(step, args.steps, stream, dev)
    x.check(stream, "after the absorbing step")
    dec_bytes, dec_flops = algorithmic_work(b)
    dec_bytes -= Bn * H * 512 * 2                     # bf16 output instead of fp32
    head_bytes = 2 * H * 128 * 512 * 2 + Bn * H * (128 * 2 + 512 * 2) + Bn * H * (512 * 2 + 128 * 4)
    app_bytes = Bn * (576 * 2 * 2 + 4)
    bytes_alg = dec_bytes + head_bytes + app_bytes
    flops = dec_flops + 4 * Bn * H * 128 * 512
    t = max(bytes_alg / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12)) * 1e6
    return {"us": ms * 1e3, "decode_step_us": decode_step_ms * 1e3, "roofline_us": t, "frac": t / (ms * 1e3),
            "algorithmic_bytes": bytes_alg,
            "note": "absorb (q_pre . w_kc) + append (one row per request) + decode + merge (bf16 out) + project "
                    "(o_lat . w_vc, fp32 out) per step, each launch a programmatic dependent of the one before; "
                    "K steps as one CUDA-graph replay over the rotating input sets; synthetic weights"}


def roofline_of(batch, peaks, peak_src, kernel_ms, step_ms):
    """The decode kernel against the roofline of this workload's algorithmic
    bytes and flops (the slower of the two at the measured peaks)."""
    bytes_alg, flops_alg = algorithmic_work(batch)
    t_hbm = bytes_alg / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops_alg / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        achieved = bytes_alg / (kernel_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    else:
        achieved = flops_alg / (kernel_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"]}
    kernel = "swab" if batch.heads <= 32 else "pair"
    roof["traffic"] = ncu_traffic(batch.spec.name if batch.spec else "custom", kernel)
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured" else "fallback"
    roof["kernel"] = f"mla_decode ({kernel})"
    roof["kernel_ms"] = kernel_ms
    roof["kernel_timing"] = "decode launches alone (no merge), rotating the input sets, one CUDA-graph replay"
    roof["algorithmic_bytes"] = bytes_alg
    roof["algorithmic_flops"] = flops_alg
    roof["roofline_us"] = max(t_hbm, t_tc) * 1e6
    roof["step_frac_of_roofline"] = max(t_hbm, t_tc) * 1e3 / step_ms
    return roof


def measure_config(batch, dev, args, peaks, peak_src, legs=()):
    """A workload besides the headline one, from the same run: its step
    (decode + merge) and its decode kernel alone, each timed as one CUDA-graph
    replay of K launches over the rotating input sets, plus the side legs
    named in `legs`."""
    import torch
    stream = torch.cuda.current_stream(dev)
    x = DecodeInputs(batch, dev, args)
    for k in range(max(args.warmup, x.R)):
        x.step(k, stream)
    x.check(stream, "after warm-up")
    step_ms = graph_ms_per_call(x.step, args.steps, stream, dev)
    kernel_ms = graph_ms_per_call(x.attend, args.steps, stream, dev)
    x.check(stream, "after timing")
    roof = roofline_of(batch, peaks, peak_src, kernel_ms, step_ms)
    absorbing = time_absorbing_step(x, dev, args, peaks, step_ms) if "absorbing_step" in legs else None
    res = {"workload": batch.spec.name, "batch": batch.batch, "heads": batch.heads, "nnz": batch.nnz,
           "step_us": step_ms * 1e3, "kernel_us": kernel_ms * 1e3, "frac": roof["frac"],
           "step_frac_of_roofline": roof["step_frac_of_roofline"], "traffic": roof["traffic"],
           "roofline_us": roof["roofline_us"], "bound": roof["bound"],
           "latent_kv_gbs": batch.nnz * 1152 / (step_ms * 1e-3) / 1e9,
           "latent_kv_gbs_kernel": batch.nnz * 1152 / (kernel_ms * 1e-3) / 1e9,
           "kernel": roof["kernel"], "input_sets": x.R}
    if absorbing is not None:
        res["absorbing_step"] = absorbing
    if "fp8" in legs:
        res["fp8_cache"] = time_fp8(batch, dev, peaks, step_ms * 1e3, x.indptr_d, x.indices_d)
    if "multi_query" in legs:
        res["multi_query"] = time_multi_query(batch, dev, peaks, x.kv, x.indptr_d, x.indices_d)
    if "cascade" in legs:
        res["cascade"] = time_cascade(batch, dev, peaks)
    if "tree" in legs:
        res["tree_verify"] = time_tree(batch, dev, peaks, x.kv, x.indptr_d, x.indices_d)
    if "head_products" in legs:
        res["head_products"] = time_head_products(batch, dev, peaks)
    del x
    torch.cuda.empty_cache()
    return res


def run_ours(args, batch, world, rank, local, pg):
    import numpy as np
    import torch
    from mla_latent_kv_absorbed_gb300 import build as B
    if rank == 0:
        B.build()
    if pg is not None:
        pg.barrier()
    B.build()
    from mla_latent_kv_absorbed_gb300 import binding, workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    x = DecodeInputs(batch, dev, args)
    dec, kv, Bn, H = x.dec, x.kv, batch.batch, batch.heads
    plan_us = host_plan_us(binding, batch.kv_indptr, H, dec.plan_host.size)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    for k in range(max(args.warmup, x.R)):
        x.step(k, stream)
    x.check(stream, "after warm-up")

    # the K timed steps captured once as a CUDA graph (decode loops replay
    # graphs: no host work between the steps' launches); one untimed replay
    cap = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for k in range(args.steps):
                x.step(k, cap)
    stream.wait_stream(cap)
    graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: K back-to-back steps (one replay of the graph)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        e_start.record(stream)
        graph.replay()
        e_end.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if pg is not None:
        pg.barrier()
    x.check(stream, "after timing")
    ms = max_over_ranks(e_start.elapsed_time(e_end) / args.steps, pg, dev)
    del graph

    # ---- the decode kernel alone: K decode launches (no merge) over the same
    # rotation, one graph replay, so that it is timed like the step
    attend_ms = max_over_ranks(graph_ms_per_call(x.attend, args.steps, stream, dev), pg, dev)

    # the same K steps launched one call at a time from the host (for reference)
    torch.cuda.synchronize()
    e0h, e1h = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0h.record(stream)
    for k in range(args.steps):
        x.step(k, stream)
    e1h.record(stream)
    torch.cuda.synchronize()
    host_launched_ms = max_over_ranks(e0h.elapsed_time(e1h) / args.steps, pg, dev)

    # ---- per-step timing with an L2-flushing write before each step (for reference)
    fl = []
    for k in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        x.step(k, stream)
        e1.record(stream)
        fl.append((e0, e1))
    torch.cuda.synchronize()
    flushed_ms = max_over_ranks(statistics.mean(a.elapsed_time(b_) for a, b_ in fl), pg, dev)
    x.check(stream, "after timing")

    # ---------------------------------------------------------------- e2e
    # Public API end to end from host buffers (mla_decode_step_host): every
    # step plans on the host, copies q, indptr, indices and the plan words in,
    # runs, and copies out and lse back.
    h_qn = torch.from_numpy(np.ascontiguousarray(batch.q_nope).view(np.int16)).view(torch.bfloat16).pin_memory()
    h_qr = torch.from_numpy(np.ascontiguousarray(batch.q_rope).view(np.int16)).view(torch.bfloat16).pin_memory()
    h_ptr = torch.from_numpy(batch.kv_indptr.astype(np.int32)).pin_memory()
    h_idx = torch.from_numpy(batch.kv_indices.astype(np.int32)).pin_memory()
    pw = int(dec.plan_host.shape[0])
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(out_dtype):
        code = 0 if out_dtype == torch.float32 else 1
        stage_bytes = binding.step_staging_bytes(Bn, H, batch.nnz, pw, code)
        bufs = []
        for j in range(2):
            bufs.append(dict(plan=torch.empty(pw, dtype=torch.int32).pin_memory(),
                             staging=torch.empty(stage_bytes, dtype=torch.uint8, device=dev),
                             h_out=torch.empty((Bn, H, 512), dtype=out_dtype).pin_memory(),
                             h_lse=torch.empty((Bn, H), dtype=torch.float32).pin_memory(),
                             done=torch.cuda.Event(), in_done=torch.cuda.Event(), run_done=torch.cuda.Event()))

        def host_step(j, pipelined):
            b = bufs[j]
            binding.decode_step_host(h_qn, h_qr, h_ptr, h_idx, kv, batch.sm_scale, b["h_out"], b["h_lse"], b["plan"],
                                     b["staging"], dec.workspace, stream, s_in if pipelined else None,
                                     s_out if pipelined else None)
            b["done"].record(s_out if pipelined else stream)
            if pipelined:
                b["in_done"].record(s_in)
                b["run_done"].record(stream)

        # (1) one step at a time, everything on one stream: the latency of a step
        for _ in range(max(2, args.warmup)):
            host_step(0, False)
            bufs[0]["done"].synchronize()
        times = []
        for _ in range(args.steps):
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            host_step(0, False)
            bufs[0]["done"].synchronize()
            times.append(time.perf_counter() - t0)
        serial_us = max_over_ranks(statistics.mean(times) * 1e6, pg, dev)
        serial_out = bufs[0]["h_out"].clone()

        # (2) steps pipelined as a serving loop runs them: kernels in order on
        # the compute stream, copies in and out on their own streams, two
        # staging buffers in turn, so step k's copies in and step k-1's copies
        # out overlap the kernels (the host waits only for the step two back
        # before reusing its pinned plan buffer)
        def pipelined(n):
            for k in range(n):
                j = k % 2
                b = bufs[j]
                if k >= 2:
                    b["in_done"].synchronize()         # step k-2's plan words have left the pinned buffer
                    s_in.wait_event(b["run_done"])     # its kernels are done reading this staging buffer
                    stream.wait_event(b["done"])       # its result has been copied out of it
                host_step(j, True)
            torch.cuda.synchronize()

        pipelined(max(2, args.warmup))
        t0 = time.perf_counter()
        pipelined(args.steps)
        us = max_over_ranks((time.perf_counter() - t0) / args.steps * 1e6, pg, dev)
        ok = bool(torch.equal(bufs[0]["h_out"], serial_out) and torch.equal(bufs[1]["h_out"], serial_out))
        h2d = (h_qn.numel() * 2 + h_qr.numel() * 2 + h_ptr.numel() * 4 + h_idx.numel() * 4 + pw * 4)
        d2h = bufs[0]["h_out"].numel() * bufs[0]["h_out"].element_size() + bufs[0]["h_lse"].numel() * 4
        return us, serial_us, ok, h2d, d2h

    e2e_us, e2e_serial_us, e2e_ok, h2d, d2h = e2e_run(torch.float32)
    e2e_bf16_us, e2e_bf16_serial_us, e2e_bf16_ok, _, d2h_bf16 = e2e_run(torch.bfloat16)
    x.check(stream, "after e2e")

    if rank != 0:
        return 0
    peaks, peak_src = load_peaks()
    roof = roofline_of(batch, peaks, peak_src, attend_ms, ms)

    head_products = time_head_products(batch, dev, peaks)
    absorbing = time_absorbing_step(x, dev, args, peaks, ms)
    multi_query = time_multi_query(batch, dev, peaks, kv, x.indptr_d, x.indices_d)
    cascade = time_cascade(batch, dev, peaks)
    tree = time_tree(batch, dev, peaks, kv, x.indptr_d, x.indices_d)
    fp8 = time_fp8(batch, dev, peaks, ms * 1e3, x.indptr_d, x.indices_d)
    rotate = x.rotate
    launches = args.steps * (1 + (1 if dec.has_merge else 0))
    del x
    torch.cuda.empty_cache()

    # ---- the other workloads of the same family, from the same run
    per_config = {}
    if not args.no_per_config:
        legs_of = {2: ("fp8", "multi_query", "cascade", "tree", "head_products", "absorbing_step"),
                   3: ("fp8", "absorbing_step"), 5: ()}
        for n in (2, 3, 4, 5):
            if n == args.workload:
                continue
            b = workloads.make_workload(n)
            per_config[b.spec.name] = measure_config(b, dev, args, peaks, peak_src, legs_of.get(n, ()))
            del b

    cpu = None
    if not args.no_cpu_baseline:
        us, nreq, tok = cpu_oracle_sample(batch, args.cpu_budget_s)
        cpu = {"value": us, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
               "sample": f"first {nreq} requests ({tok} of {batch.nnz} tokens), fp64 numpy, scaled by tokens"}
    line = {
        "metric": METRIC, "value": ms * 1e3, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, random slots)",
        "config": workload_config(batch, args, rotate),
        "latent_kv_gbs": batch.nnz * 1152 / (ms * 1e-3) / 1e9 * world,
        "step_us_l2_flushed": flushed_ms * 1e3,
        "step_us_host_launched": host_launched_ms * 1e3,
        "launch": "the K timed steps are one CUDA graph (decode + merge launches per step, the input sets rotated "
                  "as above), replayed once between the events; step_us_host_launched: the same steps issued one "
                  "call at a time from Python",
        "roofline": roof,
        "per_config": per_config,
        "head_products": head_products,
        "absorbing_step": absorbing,
        "multi_query": multi_query,
        "cascade": cascade,
        "tree_verify": tree,
        "fp8_cache": fp8,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "includes": "mla_decode_step_host: host plan + pinned H2D (q, indptr, indices, plan) + kernels + D2H "
                            "(out fp32, lse) every step; steps pipelined with copies on copy-in / copy-out streams and "
                            "two staging buffers (value), one at a time on one stream (serial_us)",
                "serial_us": e2e_serial_us, "pipelined_result_matches_serial": e2e_ok,
                "bf16_out": {"value": e2e_bf16_us, "serial_us": e2e_bf16_serial_us, "d2h_bytes_per_step": int(d2h_bf16),
                             "pipelined_result_matches_serial": e2e_bf16_ok,
                             "note": "the same loop with the output written and copied back as bf16"}},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "plan_us_host": plan_us,
        "wall_s_timed": wall,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the chosen workload (per_config stays empty)")
    ap.add_argument("--sets", type=int, default=0,
                    help="input sets rotated over the back-to-back steps (0: enough to defeat L2; 1 for profiling)")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local, pg = dist_setup(args)
    from mla_latent_kv_absorbed_gb300 import workloads
    batch = workloads.make_workload(args.workload)
    if args.impl == "reference":
        return run_reference(args, batch, rank, pg)
    return run_ours(args, batch, world, rank, local, pg)


if __name__ == "__main__":
    sys.exit(main())
