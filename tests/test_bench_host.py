"""bench.py host logic on CPU: the kernel-source hash that keeps the committed
DRAM-traffic figures tied to the code they were measured on, and the lookup
that drops them once the code differs."""

import json
import os

import bench


def test_code_only_strips_comments_and_spacing():
    src = 'int a = 1; // note\n/* block\n   comment */ const char *s = "// kept";\n\n  x  =  2 ;\n'
    assert bench._code_only(src) == 'int a = 1;\nconst char *s = "// kept";\nx = 2 ;'


def test_code_only_keeps_code_changes_visible():
    a = "if (x < 4) y = 1; // four\n"
    assert bench._code_only(a) == bench._code_only(a.replace("// four", "// 4 (comment edit)"))
    assert bench._code_only(a) != bench._code_only(a.replace("x < 4", "x < 5"))
    assert bench._code_only("a = '/';\nb = 2;") == "a = '/';\nb = 2;"


def test_traffic_figures_match_current_kernel_code():
    # The committed figures were taken on the kernels in the tree; once the
    # code changes, ncu_traffic returns None rather than a stale number.
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")) as fh:
        rec = json.load(fh)
    assert {e["source_hash"] for e in rec.values()} == {bench.kernel_source_hash()}
    T = 131072
    for kernel in ("gather", "fuse"):
        assert bench.ncu_traffic(kernel, "large", T) == rec[kernel]["bytes_per_token"] * T
        assert bench.ncu_traffic(kernel, "prefill", T) is None  # measured on one workload only
