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


def test_traffic_figures_are_used_only_for_the_code_they_were_taken_on(tmp_path, monkeypatch):
    """ncu_traffic returns a committed DRAM-traffic figure only while the
    kernel code hash it was captured at matches the tree's, and only for its
    workload and row layout; otherwise None (the bench line then reports
    traffic: null rather than a stale number)."""
    (tmp_path / "profiles").mkdir()
    T = 131072
    rec = {"gather": {"bytes_per_token": 19000, "workload": "large", "layout": "separate",
                      "source_hash": bench.kernel_source_hash()},
           "fuse": {"bytes_per_token": 18000, "workload": "large", "layout": "separate",
                    "source_hash": "0000000000000000"}}
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["gather"]["source_hash"])
    assert bench.ncu_traffic("gather", "large", T) == 19000 * T
    assert bench.ncu_traffic("gather", "prefill", T) is None  # another workload
    assert bench.ncu_traffic("gather", "large", T, layout="mx") is None  # another layout
    assert bench.ncu_traffic("fuse", "large", T) is None  # captured on other kernel code


def test_committed_traffic_figures_name_a_source_hash():
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")) as fh:
        rec = json.load(fh)
    for e in rec.values():
        assert len(e["source_hash"]) == 16 and e["bytes_per_token"] > 0 and e["command"].startswith("ncu ")
