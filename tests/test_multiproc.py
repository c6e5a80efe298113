"""The N > 1 path on CPU with world_size 2 over gloo: the bench's max-over-ranks
timing reduction and plan replicas (every rank plans the same batch: the path
shards by request with no exchange), and the reference arm under torchrun
(rank 0 alone prints its JSON line, the other rank exits 0 without output)."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    from mla_latent_kv_absorbed_gb300 import workloads as W
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # each rank times its own replica; the reported time is the slowest rank's
        mx = bench.max_over_ranks(10.0 + rank * 5.0, dist)
        # every rank builds the same synthetic batch and the same host plan words
        bt = W.make_workload(1)
        from oracle import plan_ref
        words = plan_ref.build_plan(bt.kv_indptr, bt.heads, 152)[0]
        np.save(os.path.join(out_dir, f"plan{rank}.npy"), np.asarray(words, dtype=np.int32))
        with open(os.path.join(out_dir, f"max{rank}.txt"), "w") as f:
            f.write(repr(mx))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_plan_replicas_gloo(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        assert float(open(tmp_path / f"max{r}.txt").read()) == 15.0
    assert np.array_equal(np.load(tmp_path / "plan0.npy"), np.load(tmp_path / "plan1.npy"))


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "1", "--steps", "1", "--warmup", "3",
           "--reference-budget-s", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=240, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0
