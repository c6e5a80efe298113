"""Host-side pieces of bench.py (no GPU): the code-only source digest that
keys the committed ncu traffic figures, and the form of that file."""
import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_digest_ignores_comments_and_blank_lines_only():
    a = 'int a = 1;  // one\n/* two\n   lines */\nasm("x // not a comment");\n'
    b = '\n\nint a = 1;\n// other words\nasm("x // not a comment");   /* trailing */\n'
    c = 'int a = 2;  // one\nasm("x // not a comment");\n'
    d = 'int a = 1;\nasm("x // a different literal");\n'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert bench._code_only(a) != bench._code_only(d)
    assert '"x // not a comment"' in bench._code_only(a)


def test_traffic_file_entries_are_well_formed():
    rows = []
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(line.split())
    assert rows
    for workload, kernel, nbytes, digest in rows:
        assert kernel in bench.KERNEL_SOURCES
        assert float(nbytes) > 0
        assert re.fullmatch(r"[0-9a-f]{16}", digest)
        assert len(bench.kernel_source_sha(kernel)) == 16


def test_cascade_leg_index_arrays_match_their_kv_indptr():
    # the shared-prefix leg's CSR arrays for every few-heads workload: each
    # index array holds exactly the slots its kv_indptr names, all in the pool
    from types import SimpleNamespace

    import numpy as np
    from mla_latent_kv_absorbed_gb300 import workloads as W
    for number, spec in W.WORKLOADS.items():
        if spec.heads > 32:
            continue
        rng = np.random.default_rng(spec.seed)
        lengths = W.draw_lengths(spec, rng)
        indptr = np.zeros(len(lengths) + 1, dtype=np.int32)
        indptr[1:] = np.cumsum(lengths)
        nnz = int(indptr[-1])
        batch = SimpleNamespace(batch=len(lengths), heads=spec.heads, pool=spec.pool, kv_indptr=indptr,
                                kv_indices=rng.permutation(spec.pool)[:nnz].astype(np.int32), nnz=nnz)
        c = bench.cascade_csr(batch)
        assert c["prefix_rows"] == min(4096, spec.pool)
        assert len(np.unique(c["p_ind"][:c["prefix_rows"]])) == c["prefix_rows"]
        assert len(c["p_ind"]) == c["p_ptr"][-1] and len(c["f_ind"]) == c["f_ptr"][-1]
        assert c["s_ptr"][-1] == nnz and len(c["s_ptr"]) == c["padded_batch"] + 1
        assert np.all(np.diff(c["f_ptr"]) == np.diff(c["s_ptr"]) + c["prefix_rows"])
        for a in (c["p_ind"], c["f_ind"]):
            assert a.min() >= 0 and a.max() < spec.pool


def test_topk_tree_parents_is_a_valid_breadth_first_tree():
    # the bench's draft tree: a parent before its children, top-2 fan-out,
    # drafts of depth 1..4 for eight drafts
    from oracle import mla_oracle as O
    import bench
    par = bench.topk_tree_parents(8)
    anc = O.tree_ancestors(par)
    assert par == [-1, 0, 0, 1, 1, 2, 2, 3]
    assert [len(a) for a in anc] == [1, 2, 2, 3, 3, 3, 3, 4]
    assert all(par.count(i) <= 2 for i in range(8))
