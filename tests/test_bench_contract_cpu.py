"""bench.py's host-side contract, checked without a GPU.

* `--impl reference` (the fp64 oracle timed on the host cores) prints one JSON
  line with the keys every bench line carries, plus its own `impl`,
  `cpu_baseline` and a zero-copy `e2e`.
* The source hash that attaches the committed DRAM counters to a build
  ignores comments and blank space but not code, and covers the GEMM
  kernel's sources only.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config"}


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d)
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["config"]["workload"] == "tiny"
    assert d["value"] > 0 and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "linear_cross_entropy_ce_gb300" / "csrc"
    src.mkdir(parents=True)
    f = src / "flce_gemm.cu"
    f.write_text("// header\n__global__ void k(int* p) {\n  p[0] = 1;  // one\n}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_sources_sha1()
    f.write_text("/* a new\n   comment */\n__global__   void k(int* p) {   p[0] = 1; }\n")
    assert bench.kernel_sources_sha1() == h0
    f.write_text("__global__ void k(int* p) { p[0] = 2; }\n")
    h1 = bench.kernel_sources_sha1()
    assert h1 != h0
    (src / "flce_aux.cu").write_text("__global__ void other() {}\n")   # another kernel's source
    assert bench.kernel_sources_sha1() == h1


def test_committed_traffic_matches_committed_kernel():
    sys.path.insert(0, ROOT)
    import bench
    tj = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert tj["workload"] == "llama3_8b_head"
    if tj.get("kernel_sources_sha1") != bench.kernel_sources_sha1():
        pytest.skip("kernel sources changed since the DRAM counters were taken (bench reports traffic: null)")
    assert tj["dram_bytes_per_launch"] > 0
