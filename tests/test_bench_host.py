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
