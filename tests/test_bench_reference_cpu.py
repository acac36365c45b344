"""bench.py's reference arm runs on the host alone: the float64 oracle timed on
the host cores, printing the benchmark's JSON line with impl = reference (no
GPU, no CUDA library needed)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "scan_f32_b2_L256_d16", "--steps", "2", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "elems/s"
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 3
    assert d["config"]["workload"] == "scan_f32_b2_L256_d16"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["h2d_bytes_per_step"] == 0
    assert e2e["d2h_bytes_per_step"] == 0


def test_output_check_statistics():
    """The bench's output check: relative L2 and max |err| / (1 + |ref|)."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    ref = np.array([1.0, -2.0, 0.0, 4.0])
    got = ref + np.array([0.0, 0.5, 0.1, 0.0])
    c = bench.output_check(got, ref)
    assert c["elements"] == 4
    assert abs(c["rel_l2"] - np.sqrt(0.26) / np.sqrt(21.0)) < 1e-15
    assert abs(c["max_scaled_err"] - 0.5 / 3.0) < 1e-15
    assert bench.output_check(ref, ref)["rel_l2"] == 0.0
