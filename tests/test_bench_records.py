"""The bench's committed profiler records (host logic, CPU): the ncu traffic and the per-M
tensor-pipe counters are reported only while the kernel sources still digest to the code
they were captured on, and the digest ignores comments and blank lines but not code."""

import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_records_follow_the_committed_kernel_code():
    """Reported exactly when the sources digest to the captured code, with the file's values."""
    traffic = json.load(open(os.path.join(ROOT, "profiles", "moe_traffic.json")))
    if bench.kernel_code_digest(traffic["sources"]) == traffic["code_sha256"]:
        assert bench.moe_traffic(42, 1) == 42 * traffic["dram_bytes_per_layer_m1"]
    else:
        assert bench.moe_traffic(42, 1) is None
    tp_meta = json.load(open(os.path.join(ROOT, "profiles", "moe_tensor_pipe.json")))
    assert set(tp_meta["per_m"]) == {"1", "2", "4", "8", "16", "32"}
    assert all(0.0 < r["tensor_pipe_pct"] < 100.0 for r in tp_meta["per_m"].values())
    tp = bench.tensor_pipe_per_m()
    if bench.kernel_code_digest(tp_meta["sources"]) == tp_meta["code_sha256"]:
        assert tp is not None and tp["per_m"] == tp_meta["per_m"]
    else:
        assert tp is None


def test_traffic_is_only_for_the_captured_window():
    assert bench.moe_traffic(42, 4) is None


def test_records_are_withheld_once_the_code_changes(monkeypatch):
    monkeypatch.setattr(bench, "kernel_code_digest", lambda paths: "0" * 64)
    assert bench.moe_traffic(42, 1) is None
    assert bench.tensor_pipe_per_m() is None


def test_digest_ignores_comments_but_not_code(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "a.cu").write_text("int f() {\n  return 1;  // one\n}\n")
    base = bench.kernel_code_digest(["a.cu"])
    (tmp_path / "a.cu").write_text("/* header */\nint f() {\n\n  return 1;  // uno\n}\n")
    assert bench.kernel_code_digest(["a.cu"]) == base
    (tmp_path / "a.cu").write_text("int f() {\n  return 2;\n}\n")
    assert bench.kernel_code_digest(["a.cu"]) != base
