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
    # the CUDA arm builds its config from the same workload, step and world size
    sys.path.insert(0, ROOT)
    import bench

    assert d["config"] == bench.arm_config("up", 4096, 18432, 7168, 1, ["weight_quant", "act_quant", "gemm"], 1)
    assert bench.step_kernels("up") == ["weight_quant", "act_quant", "gemm"]
    assert bench.step_kernels("decode") == ["act_quant", "gemm"]
    assert bench.step_kernels("grouped") == ["weight_quant", "act_quant", "grouped_gemm"]
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


def test_stamp_intervals_split_the_steps():
    """Each kernel's share is the interval ending at its own timestamp,
    averaged over the steps; the shares add up to the stamped step."""
    sys.path.insert(0, ROOT)
    import bench

    kernels = ["weight_quant", "act_quant", "gemm"]
    # two steps: 64, 17, 425 us and 66, 15, 427 us after a first stamp at 1000 ns
    t = [1000]
    for us in (64, 17, 425, 66, 15, 427):
        t.append(t[-1] + us * 1000)
    per, step_ms = bench.stamp_intervals(t, kernels, 2)
    assert per == {"weight_quant": 0.065, "act_quant": 0.016, "gemm": 0.426}
    assert abs(step_ms - sum(per.values())) < 1e-12
    import pytest

    with pytest.raises(ValueError):
        bench.stamp_intervals(t[:-1], kernels, 2)


def test_clock_summary_from_samples():
    """Median SM clock, minimum and the throttle reasons seen between the
    region's host times, from (time, MHz, reason bits) samples."""
    sys.path.insert(0, ROOT)
    import bench

    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.samples = [(0.0, 1000.0, 0), (1.0, 2032.0, 0), (2.0, 2010.0, 0x4), (3.0, 1990.0, 0), (9.0, 500.0, 0x40)]
    cs.max_mhz, cs.nv, cs.error = 2032.0, object(), None
    out = cs.summary(0.5, 3.5, ms=10.0)
    assert out["sm_mhz"] == 2010.0 and out["sm_mhz_min"] == 1990.0 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"] and out["region_ms_x_median_mhz"] == 20100.0
    assert cs.summary(4.0, 5.0)["reasons"] == ["unsampled"]


def test_reference_arm_under_two_ranks():
    """Launched as the multi-GPU run is (torchrun, two ranks): rank 0 alone
    times the oracle and prints the one JSON line, with n_gpus = 2; the other
    rank exits 0 without work."""
    import socket

    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
                          "--master-addr", "127.0.0.1", "--master-port", str(port),
                          os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["config"]["parallelism"] == "replicas x2"
