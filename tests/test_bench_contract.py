"""bench.py's reference arm on the CPU: one JSON line with the contract's
keys, the oracle timed on this host's cores, and an end-to-end block with no
host-device traffic.  (The CUDA arm needs a GPU and is exercised there.)"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["unit"] == "TFLOP/s" and d["data"] == "synthetic"
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_gemm_launch_count_mirrors_the_launcher():
    """The launch count bench.py claims: the up-projection GEMM never splits
    (42 tail tiles on 74 resident pairs), the down projection does (4 of
    448), the decode and tiny shapes do not; 2048 x 2560 x 6144 splits (the
    split-tail parity test's shape)."""
    sys.path.insert(0, ROOT)
    import bench

    assert bench.gemm_kernel_launches(4096, 18432, 7168, 148) == 1
    assert bench.gemm_kernel_launches(4096, 7168, 18432, 148) == 2
    assert bench.gemm_kernel_launches(64, 18432, 7168, 148) == 1
    assert bench.gemm_kernel_launches(128, 256, 256, 148) == 1
    assert bench.gemm_kernel_launches(2048, 2560, 6144, 148) == 2
    assert bench.gemm_kernel_launches(64, 7168, 18432, 148) == 2
