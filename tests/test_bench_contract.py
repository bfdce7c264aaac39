"""Host-side checks of bench.py: the reference arm's JSON line carries the
contract's keys, and a captured DRAM-traffic figure is keyed on the kernel's
code (comment edits keep it; code edits drop it)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl")


def test_reference_arm_line_has_the_contract_keys():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "w4a16_tiny",
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, OMP_NUM_THREADS="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for k in KEYS:
        assert k in line, k
    assert line["warmup"] >= 3 and line["n_gpus"] == 1 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["config"]["workload"].startswith("w4a16_tiny: w4a16_16x512x512")


def test_code_hash_ignores_comments_only():
    src = "int f(int a) {  // add one\n  /* block\n comment */ return a + 1;\n}\n"
    same = "// header\nint f(int a) {\n\n  return a + 1;  // still one\n}\n"
    other = "int f(int a) {\n  return a + 2;\n}\n"
    assert bench.code_sha256(src) == bench.code_sha256(same)
    assert bench.code_sha256(src) != bench.code_sha256(other)


def test_captured_traffic_only_for_known_calls():
    assert bench.captured_traffic("no_such_call") is None
    for name, t in bench.CAPTURED_TRAFFIC.items():
        assert t["bytes"] > 0 and t["sources"]
        for rel in t["sources"]:
            assert os.path.exists(os.path.join(ROOT, rel))


def test_sources_hash_tracks_every_source(tmp_path, monkeypatch):
    """A capture is dropped when any of its sources changes code."""
    a, b = tmp_path / "a.cu", tmp_path / "b.cuh"
    a.write_text("int f() { return 1; }\n")
    b.write_text("int g() { return 2; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.sources_sha256(["a.cu", "b.cuh"])
    monkeypatch.setitem(bench.CAPTURED_TRAFFIC, "probe_call", {"bytes": 10, "sources": ["a.cu", "b.cuh"], "sha256": h})
    assert bench.captured_traffic("probe_call") == 10
    b.write_text("// comment only\nint g() { return 2; }\n")
    assert bench.captured_traffic("probe_call") == 10
    b.write_text("int g() { return 3; }\n")
    assert bench.captured_traffic("probe_call") is None
