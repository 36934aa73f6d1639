#!/usr/bin/env python3
"""Benchmark of the fine-grained FP8 block-scaled linear layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config up|down|grouped|decode|tiny]
                    [--impl ours|reference] [--no-e2e] [--no-cpu-baseline]
    python bench.py --rows [--only TEXT] [--no-cpu-baseline]   (each kernel alone)

One step is one pass of the whole hot path over one batch of synthetic input
already resident in HBM:
  * up / down / tiny : 1x128 activation quantisation of X, 128x128 weight
                       quantisation of W, block-scaled GEMM -> Y (BF16);
  * grouped          : the same over 64 expert row groups, grouped GEMM;
  * decode           : activation quantisation + GEMM (W quantised once,
                       before timing, as the workload specifies, and packed
                       into the GEMM's stage images then as well).
The default workload is the up-projection X[4096, 7168] x W[18432, 7168].

Printed (rank 0, one JSON line): whole-job TFLOP/s (2MNK per step, all
ranks, the step's quantisation included), per-kernel times, the
roofline of the dominant kernel against the measured peaks, SM clocks sampled
during the timed region, an end-to-end figure through the C ABI with pinned
host buffers (host->device inputs and device->host Y inside the timed
region), and the CPU oracle timed on a bounded sample (rank 0, N = 1).

With --impl reference the CPU oracle itself is timed, one bounded sample of
the workload per step, on this host's cores (rank 0 only).

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and
torch.cuda.synchronize(), timed by CUDA events on the launching stream; the
maximum over ranks is reported.  The K steps are replayed from a CUDA graph
of their C-ABI calls (--no-graph: stream launches); a short device-side busy
wait before the start event covers the host's launch of the region, so the
events time the K steps alone.  Per-kernel times come
from two more passes: K stream-launched steps with a CUDA event after every
kernel (us_events: each includes the full launch gap that the event puts
before its kernel), and the K steps as a graph with a device-timestamp kernel
after every kernel (us_in_step: each kernel's share of the step as the graph
runs it, plus one short launch for the stamp).  No L2 flush:
every step's working set (inputs, codes, scales, output) is several times the
126 MB L2.  Multi-GPU runs are independent replicas (weak scaling): the
linear layer needs no exchange between ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from fp8_fine_grained_14_b300 import workloads  # noqa: E402

PROFILES = os.path.join(ROOT, "profiles")
ATTRIBUTION_IDLE_S = 0.3  # idle time before the timestamp attribution pass
HOLD_BEFORE_REGION_US = 500  # device busy wait that covers the host's launch of the timed region
CSRC = os.path.join(ROOT, "fp8_fine_grained_14_b300", "csrc")

# Dense FP8 tensor peak = measured BF16 peak x 2 (nominal dense ratio on B300:
# 4.5 PFLOP/s FP8 vs 2.25 PFLOP/s BF16).
FP8_PER_BF16 = 2.0
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# Nominal (spec-sheet) B300 figures, reported beside the measured-peak
# fractions: dense FP8 tensor rate and HBM3e bandwidth.
NOMINAL = {"fp8_tflops": 4500.0, "hbm_gbs": 8000.0}

WORKLOAD_TEXT = {
    "tiny": "tiny linear: X bf16 [128,256] ~N(0,1), W bf16 [256,256] ~N(0,0.02); "
            "1x128 act quant + 128x128 weight quant + block-scaled GEMM -> Y bf16 [128,256]",
    "up": "up-projection: X bf16 [4096,7168] ~N(0,1), W bf16 [18432,7168] ~N(0,0.02); "
          "1x128 act quant + 128x128 weight quant (E4M3, FP32 scales) + FP32-promoted block-scaled "
          "GEMM -> Y bf16 [4096,18432]",
    "down": "down-projection with outliers: X bf16 [4096,18432] ~N(0,1) with 18 channels x100, "
            "W bf16 [7168,18432] ~N(0,0.02); act + weight quant + block-scaled GEMM -> Y bf16 [4096,7168]",
    "grouped": "grouped MoE GEMM: 8192 tokens x top-8 over 64 experts (65536 rows), X bf16 [65536,7168], "
               "W bf16 [64,2048,7168]; act + weight quant + grouped block-scaled GEMM",
    "decode": "decode-shaped skinny GEMM: X bf16 [64,7168] ~N(0,1), W [18432,7168] pre-quantised 128x128 "
              "E4M3 and pre-packed into stage images; act quant + block-scaled GEMM (packed W)",
}


# ---------------------------------------------------------------------------
# Algorithmic work per kernel launch (each operand read once, each output
# written once; re-reads caused by tiling are not counted).
# ---------------------------------------------------------------------------
def step_launches(step, num_sms):
    """Kernel launches of one step: one per kernel of the step, and the dense
    GEMM's split-K reduction when it runs (not on packed weights)."""
    n = len(step.kernels)
    if step.kernels[-1] == "gemm" and step.wp is None:
        n += gemm_kernel_launches(step.M, step.N, step.K, num_sms) - 1
    return n


def gemm_kernel_launches(M, N, K, num_sms):
    """Kernels that one dense fp8_blockscaled_gemm call launches: the GEMM, and
    the split-K reduction when the launcher cuts its last round of tiles.
    Mirrors the launcher's rule: 256-column tiles on CTA pairs when the grid
    fills the GPU (128 x 128 single-CTA tiles otherwise); tail = tiles %
    resident clusters (one pair per two SMs); a split when 2 tail <= resident
    and min(resident / tail, K / 512) >= 2."""
    m_tiles = -(-M // 128)
    if N % 256 == 0 and m_tiles * (N // 256) >= num_sms:
        cg = 2 if m_tiles >= 2 else 1
        tiles, resident = -(-m_tiles // cg) * (N // 256), num_sms // cg
    else:
        tiles, resident = m_tiles * (N // 128), num_sms
    tail = tiles % resident
    if tail == 0 or 2 * tail > resident:
        return 1
    return 2 if min(resident // tail, (K // 128) // 4) >= 2 else 1


def requant_bytes(M, K):
    """FP8-cached activation -> 1x128 tiles of its transpose: the codes read
    and written once (1 B + 1 B per element) and one FP32 scale per 128
    elements on each side."""
    return 2 * M * K + 8 * (M * K // 128)


def act_quant_bytes(M, K):
    return 2 * M * K + M * K + 4 * M * (K // 128)


def weight_quant_bytes(N, K):
    return 2 * N * K + N * K + 4 * (N // 128) * (K // 128)


def gemm_bytes(M, N, K, G=1):
    return M * K + G * N * K + 4 * M * (K // 128) + 4 * G * (N // 128) * (K // 128) + 2 * M * N


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK}, "measured"
    except (OSError, ValueError, KeyError):
        return dict(FALLBACK), "fallback"


def source_digest(files):
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "gemm": ["gemm.cu", "ptx.cuh"],
    "grouped_gemm": ["gemm.cu", "ptx.cuh"],
    "act_quant": ["quant.cu", "quant_common.cuh", "ptx.cuh"],
    "weight_quant": ["quant.cu", "quant_common.cuh", "ptx.cuh"],
}


def profiled_traffic(kernel, config):
    """DRAM bytes per launch from a committed ncu summary of this kernel and
    workload, or None when there is none or the kernel source has changed
    since the counters were taken.  Summaries carry lines
    `kernel: <k>`, `config: <c>`, `source_sha256_16: <digest>` and
    `dram_bytes_per_launch: <bytes>`."""
    if not os.path.isdir(PROFILES):
        return None
    want = source_digest(KERNEL_SOURCES[kernel])
    for name in sorted(os.listdir(PROFILES)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(PROFILES, name)) as f:
            text = f.read()
        fields = dict(re.findall(r"^\s*[-*]?\s*`?(kernel|config|source_sha256_16|dram_bytes_per_launch)`?:\s*`?([\w.+-]+)`?",
                                 text, flags=re.M))
        if fields.get("kernel") == kernel and fields.get("config") == config:
            if fields.get("source_sha256_16") == want and "dram_bytes_per_launch" in fields:
                return int(float(fields["dram_bytes_per_launch"]))
    return None


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes):
    SM clock, maximum SM clock and the current clock event reasons."""

    SM = 1  # NVML_CLOCK_SM

    def __init__(self, device):
        import ctypes

        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        rc = self.lib.nvmlInit_v2()
        if rc != 0:
            raise OSError(f"nvmlInit_v2 returned {rc}")
        self.handle = ctypes.c_void_p()
        rc = -1
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            rc = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.handle))
        except Exception:
            rc = -1
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device.index), ctypes.byref(self.handle))
        if rc != 0:
            raise OSError(f"no NVML handle for {device} ({rc})")
        self._reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self._u = ctypes.c_uint()
        self._ull = ctypes.c_ulonglong()

    def clock(self, fn="nvmlDeviceGetClockInfo"):
        rc = getattr(self.lib, fn)(self.handle, self.SM, self.ct.byref(self._u))
        if rc != 0:
            raise OSError(f"{fn} returned {rc}")
        return float(self._u.value)

    def reasons(self):
        rc = self._reasons_fn(self.handle, self.ct.byref(self._ull))
        if rc != 0:
            raise OSError(f"clock event reasons: {rc}")
        return int(self._ull.value)

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """Samples the SM clock and the clock event reasons of one GPU through
    NVML (read-only queries) from a host thread, as fast as NVML answers
    (plus `period_s`), while the host waits for the timed region.  A 10 ms
    region gets tens of samples (nvidia-smi's loop is 20 ms at best)."""

    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, device, period_s=0.0002):
        import threading

        self.samples = []  # (host time, sm_mhz, reasons bitmask)
        self.max_mhz = None
        self.error = None
        self.period_s = period_s
        self._stop = threading.Event()
        self._thread = None
        try:
            self.nv = _Nvml(device)
            self.max_mhz = self.nv.clock("nvmlDeviceGetMaxClockInfo")
        except Exception as e:  # no NVML: report unsampled
            self.error = f"{type(e).__name__}: {e}"
            self.nv = None

    def _run(self):
        while not self._stop.is_set():
            try:
                mhz, reasons = self.nv.clock(), self.nv.reasons()
            except Exception as e:  # pragma: no cover
                self.error = f"{type(e).__name__}: {e}"
                return
            self.samples.append((time.perf_counter(), mhz, reasons))
            if self.period_s:
                time.sleep(self.period_s)

    def start(self):
        import threading

        if self.nv is None:
            return
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()
        t0 = time.perf_counter()
        while not self.samples and time.perf_counter() - t0 < 1.0:  # first sample before the region starts
            time.sleep(0.0001)

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self.nv is not None:
            try:
                self.nv.close()
            except Exception:
                pass

    def summary(self, t0=None, t1=None, ms=None):
        """Samples between host times t0 and t1 (the timed region): median SM
        MHz, the maximum SM clock, the reasons seen, and the region's time x
        median MHz (cycles at the median clock)."""
        sel = [s for s in self.samples if (t0 is None or s[0] >= t0) and (t1 is None or s[0] <= t1)]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0,
                    "source": "nvml" if self.nv is not None else f"unavailable ({self.error})"}
        seen = sorted(name for name, bit in self.REASONS.items() if any(r & bit for _, _, r in sel))
        med = statistics.median(m for _, m, _ in sel)
        out = {"sm_mhz": med, "sm_max_mhz": self.max_mhz, "sm_mhz_min": min(m for _, m, _ in sel),
               "reasons": seen, "samples": len(sel), "source": "NVML (read-only) polled from a host thread"}
        if ms is not None:
            out["region_ms_x_median_mhz"] = ms * med
        return out


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas; the barrier and max-over-ranks only)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group(backend=backend)
        return dist
    return None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value, device):
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# Workload setup
# ---------------------------------------------------------------------------
def make_inputs(name, seed):
    """CPU tensors of the workload (seeded; see fp8_fine_grained_14_b300.workloads)."""
    if name == "grouped":
        c = workloads.CONFIGS["grouped"]
        offsets, x, w = workloads.grouped_inputs(**{k: c[k] for k in ("tokens", "topk", "G", "N", "K")}, seed=seed)
        return {"offsets": offsets, "x": x, "w": w}
    x, w = workloads.config_inputs(name, seed=seed)
    return {"x": x, "w": w}


def shapes(name, inp):
    if name == "grouped":
        G, N, K = inp["w"].shape
        return dict(M=inp["x"].shape[0], N=N, K=K, G=G)
    return dict(M=inp["x"].shape[0], N=inp["w"].shape[0], K=inp["x"].shape[1], G=1)


class Step:
    """Pre-marshalled C-ABI calls of one step on one stream."""

    def __init__(self, name, inp, device, stream, fb):
        self.name = name
        self.fb = fb
        self.lib = fb.binding.lib
        self.stream = stream
        s = shapes(name, inp)
        self.M, self.N, self.K, self.G = s["M"], s["N"], s["K"], s["G"]
        M, N, K, G = self.M, self.N, self.K, self.G
        self.x = inp["x"].to(device)
        self.w = inp["w"].to(device)
        self.qa = torch.empty((M, K), dtype=torch.uint8, device=device)
        self.sa = torch.empty((K // 128, fb.ld_sa_for(M)), dtype=torch.float32, device=device)
        self.qw = torch.empty((G * N, K), dtype=torch.uint8, device=device)
        self.sw = torch.empty((G * N // 128, K // 128), dtype=torch.float32, device=device)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        self.offsets = inp["offsets"].to(device) if "offsets" in inp else None
        self.kernels = step_kernels(name)
        self.wp = None
        if name == "decode":
            # the weights are prepared before timing: quantised, then packed
            # into the GEMM's stage images so each stage streams as one
            # contiguous 16 KB copy
            with torch.cuda.stream(stream):
                self.weight_quant()
                self.wp = fb.fp8_pack_weight_128x128(self.qw, stream=stream)
            stream.synchronize()

    def _st(self):
        import ctypes

        return ctypes.c_void_p(self.stream.cuda_stream)

    def _check(self, fn, status):
        if status != 0:
            raise self.fb.Fp8bsError(fn, status)

    def act_quant(self):
        p = lambda t: t.data_ptr()  # noqa: E731
        self._check("fp8_quant_act_1x128", self.lib.fp8_quant_act_1x128(
            p(self.x), self.M, self.K, self.x.stride(0), p(self.qa), self.qa.stride(0), p(self.sa),
            self.sa.stride(0), self._st()))

    def weight_quant(self):
        p = lambda t: t.data_ptr()  # noqa: E731
        self._check("fp8_quant_weight_128x128", self.lib.fp8_quant_weight_128x128(
            p(self.w), self.G * self.N, self.K, self.K, p(self.qw), self.qw.stride(0), p(self.sw), self._st()))

    def gemm(self):
        p = lambda t: t.data_ptr()  # noqa: E731
        if self.wp is not None:
            self._check("fp8_blockscaled_gemm_packed", self.lib.fp8_blockscaled_gemm_packed(
                p(self.qa), self.qa.stride(0), p(self.sa), self.sa.stride(0), p(self.wp), p(self.sw), p(self.y),
                self.y.stride(0), self.M, self.N, self.K, self._st()))
            return
        self._check("fp8_blockscaled_gemm", self.lib.fp8_blockscaled_gemm(
            p(self.qa), self.qa.stride(0), p(self.sa), self.sa.stride(0), p(self.qw), self.qw.stride(0),
            p(self.sw), p(self.y), self.y.stride(0), self.M, self.N, self.K, self._st()))

    def grouped_gemm(self):
        p = lambda t: t.data_ptr()  # noqa: E731
        self._check("fp8_blockscaled_grouped_gemm", self.lib.fp8_blockscaled_grouped_gemm(
            self.G, p(self.offsets), self.M, p(self.qa), self.qa.stride(0), p(self.sa), self.sa.stride(0),
            p(self.qw), p(self.sw), p(self.y), self.y.stride(0), self.N, self.K, self._st()))

    def run(self, events=None, stamps=None):
        """One step; if `events` is a list, an event is recorded after each
        kernel; if `stamps` is a DeviceStamps, a device timestamp is enqueued
        after each kernel."""
        for k in self.kernels:
            getattr(self, k)()
            if events is not None:
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(self.stream)
                events.append(ev)
            if stamps is not None:
                # after the act quantiser the stamp passes on its early release
                stamps.mark(self.stream, release_next=(k == "act_quant"))

    def flops(self):
        return 2 * self.M * self.N * self.K

    def algorithmic(self, kernel):
        M, N, K, G = self.M, self.N, self.K, self.G
        if kernel == "act_quant":
            return act_quant_bytes(M, K), "hbm"
        if kernel == "weight_quant":
            return weight_quant_bytes(G * N, K), "hbm"
        if self.name == "decode":
            return gemm_bytes(M, N, K), "hbm"
        return 2 * M * N * K, "tensor"


class DeviceStamps:
    """Device-side timestamps (ns of the GPU's global timer) written by the
    library's fp8bs_stream_timestamp kernel, which starts once the kernel
    before it has completed.  Unlike an event record it keeps the step's
    kernels programmatic dependents of one another, so the intervals between
    consecutive stamps are each kernel's share of the step as the timed graph
    runs it (plus about one short launch per stamp)."""

    def __init__(self, fb, count, device):
        self.fb = fb
        self.t = torch.zeros(count, dtype=torch.int64, device=device)
        self.i = 0

    def mark(self, stream, release_next=False):
        self.fb.fp8bs_stream_timestamp(self.t, self.i, release_next, stream)
        self.i += 1


def hold_gpu(stream, us):
    """Enqueue a device-side busy wait of about `us` microseconds."""
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None and us > 0:
        with torch.cuda.stream(stream):
            sleep(int(us * 2000))  # cycles at about 2 GHz


def capture_steps(step, stream, steps):
    """The C-ABI calls of `steps` steps recorded into one CUDA graph (the
    kernels, their arguments and their order; the library's host-side
    validation and tensor-map encoding run once, at capture).  Replaying it
    launches exactly the kernels that the stream-launched steps launch, with
    about 1 us between dependent kernels instead of the 3-6 us of separate
    stream launches.  Returns None when the calls cannot be captured."""
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            for _ in range(steps):
                step.run()
        return g
    except Exception as e:  # e.g. an allocation the capture does not accept
        torch.cuda.synchronize()
        print(f"note: the step could not be captured in a CUDA graph ({type(e).__name__}: {e}); "
              "timing stream launches", file=sys.stderr)
        return None


def time_device(step, stream, steps, warmup, dist, device, use_graph=True):
    """The timed region: `steps` steps bracketed by a barrier and a device
    synchronisation on both sides, timed by CUDA events on the launching
    stream; the steps are replayed from a CUDA graph of the same C-ABI calls
    (stream-launched when capture is unavailable or disabled).

    Per-kernel durations then come from a second pass of `steps`
    stream-launched steps with a CUDA event recorded after every kernel: a
    kernel's duration runs from the previous event to its own, so it includes
    the launch gap before the kernel (3-6 us on B300) and never understates
    the kernel."""
    for _ in range(warmup):
        with torch.cuda.stream(stream):
            step.run()
    torch.cuda.synchronize(device)
    if step.fb.fp8bs_last_device_error(stream) != 0:
        raise RuntimeError("device status word set during warm-up")
    graph = capture_steps(step, stream, steps) if use_graph else None
    launch_mode = "CUDA graph of the steps' C-ABI calls" if graph is not None else "stream launches"
    if graph is not None:
        graph.replay()  # untimed: uploads the graph
        torch.cuda.synchronize(device)
    sampler = ClockSampler(device)
    sampler.start()
    barrier(dist, device)
    torch.cuda.synchronize(device)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        # keep the GPU busy (a device-side sleep, outside the timed window)
        # while the host enqueues the start event and the graph launch, so
        # the window holds the K steps and none of the host's launch time
        hold_gpu(stream, HOLD_BEFORE_REGION_US)
        start.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for _ in range(steps):
                step.run()
        end.record(stream)
    torch.cuda.synchronize(device)
    t1 = time.perf_counter()
    barrier(dist, device)
    sampler.stop()
    total_ms = start.elapsed_time(end)
    status = step.fb.fp8bs_last_device_error(stream)
    if status != 0:
        raise RuntimeError(f"device status word {status} after the timed region")
    del graph
    # per-kernel attribution pass (stream launches: run at once, while the
    # host is still busy, so that launches keep pace)
    events = []
    a = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            step.run(events)
    torch.cuda.synchronize(device)
    nk = len(step.kernels)
    per_kernel = {k: 0.0 for k in step.kernels}
    prev = a
    for i, ev in enumerate(events):
        per_kernel[step.kernels[i % nk]] += prev.elapsed_time(ev)
        prev = ev
    per_kernel = {k: v / steps for k, v in per_kernel.items()}
    attribution_ms = a.elapsed_time(events[-1]) / steps
    status = step.fb.fp8bs_last_device_error(stream)
    if status != 0:
        raise RuntimeError(f"device status word {status} after the attribution pass")
    stamped = None
    if launch_mode.startswith("CUDA graph"):
        # one graph launch, so host speed does not matter; start it, like the
        # timed region, from a GPU that has not just run a long burst
        # (the power cap averages over a window)
        time.sleep(ATTRIBUTION_IDLE_S)
        stamped = stamp_attribution(step, stream, steps, device)
    return total_ms, per_kernel, sampler.summary(t0, t1, total_ms), attribution_ms, launch_mode, stamped


def stamp_attribution(step, stream, steps, device):
    """Per-kernel shares of the step from device timestamps: the same steps
    captured as a CUDA graph, with a timestamp kernel after every kernel (and
    one before the first), replayed once (the stamps are device times, so
    the graph's upload at its first launch precedes the first stamp).
    Returns ({kernel: ms per step}, ms per step from first to last stamp,
    SM clocks sampled during the replay), or None when the steps cannot be
    captured."""
    nk = len(step.kernels)
    st = DeviceStamps(step.fb, steps * nk + 1, device)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            st.mark(stream)
            for _ in range(steps):
                step.run(stamps=st)
    except Exception as e:
        torch.cuda.synchronize()
        print(f"note: timestamped steps could not be captured ({type(e).__name__}: {e})", file=sys.stderr)
        return None
    sampler = ClockSampler(device)
    sampler.start()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize(device)
    t1 = time.perf_counter()
    sampler.stop()
    status = step.fb.fp8bs_last_device_error(stream)
    if status != 0:
        raise RuntimeError(f"device status word {status} after the timestamp pass")
    t = st.t.cpu().tolist()
    del g
    per_kernel, step_ms = stamp_intervals(t, step.kernels, steps)
    return per_kernel, step_ms, sampler.summary(t0, t1)


def stamp_intervals(t, kernels, steps):
    """Per-kernel ms per step from the timestamps (ns) of a stamped run: t[0]
    before the first kernel, then one after each kernel of each step in
    order.  Kernel i of a step gets the interval ending at its own stamp.
    Returns ({kernel: ms per step}, ms per step from the first to the last
    stamp)."""
    nk = len(kernels)
    if len(t) != steps * nk + 1:
        raise ValueError("one timestamp before the steps and one after each kernel")
    per_kernel = {k: 0.0 for k in kernels}
    for i in range(steps * nk):
        per_kernel[kernels[i % nk]] += (t[i + 1] - t[i]) * 1e-6
    return {k: v / steps for k, v in per_kernel.items()}, (t[-1] - t[0]) * 1e-6 / steps


def time_e2e(name, inp, step, stream, steps, warmup, device, fb):
    """Same metric through the public API from pinned host buffers: per step
    the inputs go host->device and Y comes back device->host inside the timed
    region (wall clock, synchronised on both sides).  Dense workloads use the
    pipelined HostPipeline (copies of one step overlap the kernels of the
    next); the grouped workload runs its copies and kernels in sequence."""
    hx = inp["x"].pin_memory()
    hw = inp["w"].pin_memory() if name != "decode" else None
    hy = [torch.empty(step.y.shape, dtype=step.y.dtype).pin_memory() for _ in range(2)]
    h2d = hx.numel() * hx.element_size() + (hw.numel() * hw.element_size() if hw is not None else 0)
    d2h = hy[0].numel() * hy[0].element_size()

    if name == "grouped":
        def one(i):
            with torch.cuda.stream(stream):
                step.x.copy_(hx, non_blocking=True)
                step.w.copy_(hw.view(step.w.shape), non_blocking=True)
                step.run()
                hy[i % 2].copy_(step.y, non_blocking=True)

        def sync():
            stream.synchronize()
    else:
        pipe = fb.HostPipeline(step.M, step.N, step.K, device=device, depth=2,
                               prequantised_w=(step.qw, step.sw) if name == "decode" else None)

        def one(i):
            pipe.submit(hx, hw, hy[i % 2])

        def sync():
            pipe.synchronize()

    for i in range(warmup):
        one(i)
    sync()
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    sync()
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - t0
    mode = ("stream-ordered copies and calls" if name == "grouped" else
            "HostPipeline, kernels replayed from CUDA graphs" if pipe.graphed else
            f"HostPipeline, direct calls ({pipe.capture_error})")
    return wall / steps * 1e3, wall, h2d, d2h, mode


# ---------------------------------------------------------------------------
# CPU oracle timing (test infrastructure; only these legs of the benchmark
# execute the oracle).  The unchanged oracle runs row-parallel over every core
# in this process's affinity mask (oracle.parallel: one worker process per
# core, one BLAS thread each, row slices that the method keeps independent).
# ---------------------------------------------------------------------------
def oracle_threads():
    """Threads the oracle's BLAS pool uses in this process (the per-row
    timings of --rows run the oracle here, on one process)."""
    try:
        from threadpoolctl import threadpool_info

        return max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        return 1


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _bf16_bits(t):
    return t.contiguous().view(torch.int16).numpy()


class OracleSample:
    """The oracle's whole step on rows [0, m_rows) of X and the first n_rows
    (a multiple of 128) weight rows (of expert 0 when grouped), row-parallel
    over the host's cores.  The weights of the decode workload are quantised
    once, outside the timing, as the workload specifies."""

    def __init__(self, pool, name, inp):
        self.pool, self.name, self.inp = pool, name, inp
        self._preq = {}

    def run(self, m_rows, n_rows):
        x = _bf16_bits(self.inp["x"][:m_rows])
        w = self.inp["w"][0] if self.name == "grouped" else self.inp["w"]
        w = _bf16_bits(w[:n_rows])
        K = x.shape[1]
        if self.name == "decode" and n_rows not in self._preq:
            self._preq[n_rows] = self.pool.quant_weight_128x128(w)
        t0 = time.perf_counter()
        qa, sa = self.pool.quant_act_1x128(x)
        qw, sw = self._preq[n_rows] if self.name == "decode" else self.pool.quant_weight_128x128(w)
        self.pool.blockscaled_gemm(qa, sa, qw, sw)
        return time.perf_counter() - t0, 2 * m_rows * n_rows * K

    def describe(self, m_rows, n_rows):
        what = "expert 0's " if self.name == "grouped" else ""
        quant = "quantisation of X" if self.name == "decode" else "quantisation of X and W"
        return (f"CPU oracle (numpy; float64 GEMM) on X[:{m_rows}] and {what}W[:{n_rows}] with the full K: {quant} "
                f"and the block-scaled GEMM, row-parallel over {self.pool.workers} worker processes (one per core "
                f"of the {host_cores()} in this process's affinity mask, one BLAS thread each)")


def cpu_baseline(name, inp, target_s=12.0):
    from oracle.parallel import OraclePool

    M = inp["x"].shape[0]
    N = inp["w"].shape[-2]
    m_rows = min(M, 1024)
    n_rows = min(N, 2048)
    with OraclePool() as pool:
        smp = OracleSample(pool, name, inp)
        smp.run(min(M, 128), min(N, 128))  # warm the workers
        t, fl = smp.run(m_rows, n_rows)
        reps = max(1, min(20, int(target_s / max(t, 1e-3))))
        tot_t, tot_f = t, fl
        for _ in range(reps - 1):
            t, fl = smp.run(m_rows, n_rows)
            tot_t += t
            tot_f += fl
        return {
            "value": tot_f / tot_t / 1e12,
            "unit": "TFLOP/s",
            "cores": pool.workers,
            "kind": "oracle",
            "sample": f"{smp.describe(m_rows, n_rows)}; {reps} repetitions ({tot_t:.1f} s); value = sample FLOPs / "
                      f"sample time",
        }


def arm_config(name, M, N, K, G, kernels, world):
    """The `config` of the JSON line, identical for both arms."""
    return {"workload": WORKLOAD_TEXT[name], "name": name, "M": M, "N": N, "K": K, "G": G,
            "step": " + ".join(kernels), "l2": "no flush: inputs larger than L2 (step working set > 126 MB)",
            "parallelism": f"replicas x{world}"}


def step_kernels(name):
    """The kernels of one step, in order: the weights are quantised (once per
    weight update; the decode workload's weights are pre-quantised), then the
    activations online, then the GEMM."""
    return ([] if name == "decode" else ["weight_quant"]) + ["act_quant"] + \
        (["grouped_gemm"] if name == "grouped" else ["gemm"])


# ---------------------------------------------------------------------------
# Arms
# ---------------------------------------------------------------------------
def run_reference(args):
    from oracle.parallel import OraclePool

    rank, world, _ = dist_env()
    if rank != 0:
        return
    name = args.config
    inp = make_inputs(name, seed=0)
    s = shapes(name, inp)
    M, N, K, G = s["M"], s["N"], s["K"], s["G"]
    # size each step's sample so that warm-up + steps end within ~150 s
    budget = 150.0 / max(1, args.steps + args.warmup)
    with OraclePool() as pool:
        smp = OracleSample(pool, name, inp)
        n_rows = min(N, 512)
        m_rows = min(M, 16)
        t, _ = smp.run(m_rows, n_rows)
        while m_rows * 2 <= min(M, 2048) and t * 2 <= budget:
            m_rows *= 2
            t, _ = smp.run(m_rows, n_rows)
        for _ in range(args.warmup):
            smp.run(m_rows, n_rows)
        t0 = time.perf_counter()
        flops = 0
        for _ in range(args.steps):
            _, fl = smp.run(m_rows, n_rows)
            flops += fl
        elapsed = time.perf_counter() - t0
        cores = pool.workers
        sample = smp.describe(m_rows, n_rows)
    value = flops / elapsed / 1e12
    unit = "TFLOP/s"
    line = {
        "impl": "reference",
        "metric": "block-scaled FP8 GEMM TFLOPS (incl. quant) vs FP8 peak; quant GB/s vs HBM",
        "value": value, "unit": unit, "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": arm_config(name, M, N, K, G, step_kernels(name), args.gpus),
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": f"per step: {sample}; rank 0 only; value = sample FLOPs / time"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Per-row measurements: every kernel of the scope table on its own, at full
# size, against its roofline, with the CPU oracle timed on a bounded sample
# in the same unit.  One JSON line per row, apart from the step's benchmark line.
# ---------------------------------------------------------------------------
_FLUSH = None


def _time_kernel(fn, iters=40, warmup=3):
    """Time of fn() on the current stream, L2 evicted before each of `iters`
    runs: a 512 MB buffer is read (a sum), which evicts every input from L2
    without leaving dirty lines whose write-back would be charged to the
    timed call.  Returns (ms from device timestamps, ms from CUDA events),
    each the mean of the middle half of the runs.  The timestamps are
    fp8bs_stream_timestamp kernels before and after the call; the library's
    kernels launch as programmatic dependents of the first, so the interval
    is the call's kernels plus one short dependent-launch gap.  Event
    timestamps advance in steps of about 2 us here and each event interval
    also holds the full launch gap before the kernel.  Output lines still
    dirty in L2 when the call ends are written back during the next eviction
    read, so a row that writes much (E5M6: as many bytes as it reads) can
    read above the copy peak."""
    global _FLUSH
    if _FLUSH is None:
        _FLUSH = torch.ones(128 * 2 ** 20, dtype=torch.float32, device="cuda")
    fb = load_library()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stamps = torch.zeros(2 * iters, dtype=torch.int64, device="cuda")
    ts = []
    for i in range(iters):
        _FLUSH.sum()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fb.fp8bs_stream_timestamp(stamps, 2 * i)
        fn()
        fb.fp8bs_stream_timestamp(stamps, 2 * i + 1)
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    t = stamps.cpu().tolist()
    ds = [(t[2 * i + 1] - t[2 * i]) * 1e-6 for i in range(iters)]

    def middle_mean(v):
        v = sorted(v)
        mid = v[len(v) // 4: len(v) - len(v) // 4]
        return sum(mid) / len(mid)

    return middle_mean(ds), middle_mean(ts)


def _time_cpu(fn, budget_s=2.0):
    t0 = time.perf_counter()
    n = 0
    while True:
        fn()
        n += 1
        t = time.perf_counter() - t0
        if t >= budget_s or n >= 50:
            return t / n


def run_rows(args):
    import numpy as np

    import oracle  # CPU baseline only

    fb = load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_PER_BF16
    g = torch.Generator(device=dev).manual_seed(0)
    gc = torch.Generator().manual_seed(0)

    def bf16(*shape, std=1.0):
        return (torch.randn(*shape, generator=g, device=dev) * std).to(torch.bfloat16)

    def bf16c(*shape, std=1.0):
        return (torch.randn(*shape, generator=gc) * std).to(torch.bfloat16).float().numpy()

    lines = []
    sampler = ClockSampler(dev, period_s=0.001)
    sampler.start()

    def emit(row, what, timer, work, unit, oracle_fn=None, oracle_work=None, oracle_sample=""):
        if args.only and not any(t in f"{row} {what}" for t in args.only.split("|")):
            return
        t0 = time.perf_counter()
        ms, ms_events = timer()
        clocks = sampler.summary(t0, time.perf_counter())
        scale = 1e9 if unit == "GB/s" else 1e12
        peak = peaks["hbm_gbs"] if unit == "GB/s" else fp8_peak
        achieved = work / (ms * 1e-3) / scale
        line = {"row": row, "workload": what, "us": ms * 1e3, "achieved": achieved, "unit": unit, "peak": peak,
                "frac": achieved / peak, "us_events": ms_events * 1e3,
                "frac_events": work / (ms_events * 1e-3) / scale / peak, "peak_source": peak_src,
                "algorithmic": work,
                "timing": "device timestamps around the call (L2 evicted before each run); us_events: CUDA events",
                "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_mhz_min", "reasons", "samples")}}
        if oracle_fn is not None and not args.no_cpu_baseline:
            t = _time_cpu(oracle_fn)
            scale = 1e9 if unit == "GB/s" else 1e12
            line["oracle"] = {"value": oracle_work / t / scale, "unit": unit, "sample": oracle_sample,
                              "threads": oracle_threads()}
        print(json.dumps(line), flush=True)
        lines.append(line)

    M, N, K = 4096, 18432, 7168
    x, w = bf16(M, K), bf16(N, K, std=0.02)
    xs, ws = bf16c(256, K), bf16c(256, K, std=0.02)
    qa, sa = fb.fp8_quant_act_1x128(x)
    qw, sw = fb.fp8_quant_weight_128x128(w)
    emit("a1 act quant 1x128", f"X [{M},{K}] BF16", lambda: _time_kernel(lambda: fb.fp8_quant_act_1x128(x, qa=qa, sa=sa)),
         act_quant_bytes(M, K), "GB/s", lambda: oracle.quant_act_1x128(xs), act_quant_bytes(256, K), "X[:256]")
    emit("a2 weight quant 128x128", f"W [{N},{K}] BF16",
         lambda: _time_kernel(lambda: fb.fp8_quant_weight_128x128(w, qw=qw, sw=sw)), weight_quant_bytes(N, K), "GB/s",
         lambda: oracle.quant_weight_128x128(ws), weight_quant_bytes(256, K), "W[:256]")
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    qas, sas = oracle.quant_act_1x128(xs[:128])
    qws, sws = oracle.quant_weight_128x128(ws)
    emit("a3-a5 GEMM (BF16 out)", f"up {M}x{N}x{K}",
         lambda: _time_kernel(lambda: fb.fp8_blockscaled_gemm(qa, sa, qw, sw, y=y)), 2 * M * N * K, "TFLOP/s",
         lambda: oracle.blockscaled_gemm(qas, sas, qws, sws), 2 * 128 * 256 * K, "128 x 256 outputs, full K")
    y32 = torch.empty((M, N), dtype=torch.float32, device=dev)
    emit("NEXT1 GEMM (FP32 out)", f"up {M}x{N}x{K}",
         lambda: _time_kernel(lambda: fb.fp8_blockscaled_gemm(qa, sa, qw, sw, y=y32)), 2 * M * N * K, "TFLOP/s")
    del y32
    # down projection
    xd, wd = bf16(M, N), bf16(K, N, std=0.02)
    qad, sad = fb.fp8_quant_act_1x128(xd)
    qwd, swd = fb.fp8_quant_weight_128x128(wd)
    yd = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    emit("a3-a5 GEMM (BF16 out)", f"down {M}x{K}x{N}",
         lambda: _time_kernel(lambda: fb.fp8_blockscaled_gemm(qad, sad, qwd, swd, y=yd)), 2 * M * N * K, "TFLOP/s")
    rres = bf16(M, K)
    emit("NEXT1 GEMM + BF16 residual", f"down {M}x{K}x{N}, R [{M},{K}] BF16",
         lambda: _time_kernel(lambda: fb.fp8_blockscaled_gemm_residual(qad, sad, qwd, swd, rres, y=yd)),
         2 * M * N * K, "TFLOP/s")
    del rres
    # decode
    xdec = bf16(64, K)
    qdec, sdec = fb.fp8_quant_act_1x128(xdec)
    ydec = torch.empty((64, N), dtype=torch.bfloat16, device=dev)
    emit("a7 decode GEMM", f"64x{N}x{K}, W pre-quantised",
         lambda: _time_kernel(lambda: fb.fp8_blockscaled_gemm(qdec, sdec, qw, sw, y=ydec)), gemm_bytes(64, N, K), "GB/s")
    wpk = fb.fp8_pack_weight_128x128(qw)
    emit("a7 decode GEMM, packed W", f"64x{N}x{K}, W pre-quantised and packed",
         lambda: _time_kernel(lambda: fb.fp8_blockscaled_gemm_packed(qdec, sdec, wpk, sw, y=ydec)),
         gemm_bytes(64, N, K), "GB/s")
    emit("a7 weight pack", f"W codes [{N},{K}]",
         lambda: _time_kernel(lambda: fb.fp8_pack_weight_128x128(qw, wp=wpk)), 2 * N * K, "GB/s")
    del wpk
    # grouped (MoE): codes and scales drawn directly (the GEMM's inputs)
    cg = workloads.CONFIGS["grouped"]
    routes = torch.multinomial(torch.ones(cg["tokens"], cg["G"]), cg["topk"], replacement=False, generator=gc)
    offsets = workloads.grouped_offsets(torch.bincount(routes.flatten(), minlength=cg["G"])).to(dev)
    Mg, Gg, Ng = cg["tokens"] * cg["topk"], cg["G"], cg["N"]

    def codes(*shape):
        c = torch.randint(0, 0x7E, shape, generator=g, device=dev, dtype=torch.int32)
        return (c | (torch.randint(0, 2, shape, generator=g, device=dev, dtype=torch.int32) << 7)).to(torch.uint8)

    qag, qwg = codes(Mg, K), codes(Gg, Ng, K)
    sag = torch.rand((K // 128, Mg), generator=g, device=dev) * 0.01 + 1e-3
    swg = torch.rand((Gg, Ng // 128, K // 128), generator=g, device=dev) * 0.01 + 1e-3
    yg = torch.empty((Mg, Ng), dtype=torch.bfloat16, device=dev)
    emit("a6 grouped GEMM", f"{Gg} experts, {Mg} routed rows, N={Ng}, K={K}",
         lambda: _time_kernel(lambda: fb.fp8_blockscaled_grouped_gemm(offsets, Mg, qag, sag, qwg, swg, y=yg)),
         2 * Mg * Ng * K, "TFLOP/s")
    del qag, qwg, sag, swg, yg
    # dequant
    wback = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    emit("NEXT3 block dequant", f"W [{N},{K}]", lambda: _time_kernel(lambda: fb.fp8_dequant_weight_128x128(qw, sw, y=wback)),
         N * K + 2 * N * K + 4 * (N // 128) * (K // 128), "GB/s",
         lambda: oracle.dequant_weight_128x128_bf16(qws, sws), 3 * 256 * K, "W[:256]")
    del wback, xd, wd, qad, sad, qwd, swd, yd
    # backward
    qt = torch.empty((K, M), dtype=torch.uint8, device=dev)
    st = torch.empty((M // 128, K), dtype=torch.float32, device=dev)
    emit("NEXT2 act quant of X^T", f"X [{M},{K}]",
         lambda: _time_kernel(lambda: fb.fp8_quant_act_1x128_t(x, qt=qt, st=st)), act_quant_bytes(M, K), "GB/s",
         lambda: oracle.quant_act_1x128_t(bf16c(256, 1024)), act_quant_bytes(256, 1024), "X[:256, :1024]")
    qxs, sxs = oracle.quant_act_1x128(bf16c(256, 1024))
    emit("NEXT2 requant of FP8-cached X^T", f"qa [{M},{K}] + 1x128 scales -> X^T codes + scales",
         lambda: _time_kernel(lambda: fb.fp8_requant_act_1x128_t(qa, sa, qt=qt, st=st)), requant_bytes(M, K), "GB/s",
         lambda: oracle.requant_act_1x128_t(qxs, sxs), requant_bytes(256, 1024), "qa[:256, :1024]")
    qwt = torch.empty((K, N), dtype=torch.uint8, device=dev)
    swt = torch.empty((K // 128, N // 128), dtype=torch.float32, device=dev)
    emit("NEXT2 weight code transpose", f"W codes [{N},{K}]",
         lambda: _time_kernel(lambda: fb.fp8_transpose_weight_128x128(qw, sw, qwt=qwt, swt=swt)), 2 * N * K, "GB/s")
    dy = bf16(M, N)
    qdy, sdy = fb.fp8_quant_act_1x128(dy)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    emit("NEXT2 dgrad GEMM", f"dX = dY.W: {M}x{K}x{N}",
         lambda: _time_kernel(lambda: fb.fp8_blockscaled_gemm(qdy, sdy, qwt, swt, y=dx)), 2 * M * N * K, "TFLOP/s")
    qdyt, sdyt = fb.fp8_quant_act_1x128_t(dy)
    dw = torch.empty((N, K), dtype=torch.float32, device=dev)
    qat, sat = oracle.quant_act_1x128_t(bf16c(M, 128))
    qbt, sbt = oracle.quant_act_1x128_t(bf16c(M, 256))
    emit("NEXT2 wgrad GEMM (row-scaled, FP32 out)", f"dW = dY^T.X: {N}x{K}x{M}",
         lambda: _time_kernel(lambda: fb.fp8_blockscaled_gemm_rowscaled(qdyt, sdyt, qt, st, y=dw)), 2 * M * N * K,
         "TFLOP/s", lambda: oracle.blockscaled_gemm_rowscaled(qat, sat, qbt, sbt), 2 * 128 * 256 * M,
         "128 x 256 outputs, full token range")
    del qt, st, qwt, swt, dy, qdy, sdy, dx, qdyt, sdyt, dw
    # variants
    qpt = torch.empty((M, K), dtype=torch.uint8, device=dev)
    spt = torch.empty((M,), dtype=torch.float32, device=dev)
    emit("NEXT4 per-token quant", f"X [{M},{K}]", lambda: _time_kernel(lambda: fb.fp8_quant_per_token(x, q=qpt, s=spt)),
         3 * M * K + 4 * M, "GB/s", lambda: oracle.quant_per_token(xs), 3 * 256 * K, "X[:256]")
    spc = torch.empty((K,), dtype=torch.float32, device=dev)
    emit("NEXT4 per-channel quant", f"X [{M},{K}], one pass on 8-CTA clusters",
         lambda: _time_kernel(lambda: fb.fp8_quant_per_channel(x, q=qpt, s=spc)), 3 * M * K + 4 * K, "GB/s",
         lambda: oracle.quant_per_channel(xs), 3 * 256 * K, "X[:256]")
    codes = torch.empty((M, K), dtype=torch.int16, device=dev)
    emit("NEXT4 E5M6 encode", f"X [{M},{K}]", lambda: _time_kernel(lambda: fb.e5m6_encode(x, codes=codes)), 4 * M * K,
         "GB/s", lambda: oracle.e5m6_encode_rne_satfinite(xs), 4 * 256 * K, "X[:256]")
    del codes, qpt, spt, spc
    F = N
    gu = bf16(M, 2 * F, std=2.0)
    qh = torch.empty((M, F), dtype=torch.uint8, device=dev)
    sh = torch.empty((F // 128, M), dtype=torch.float32, device=dev)
    gus = bf16c(128, 2 * F, std=2.0)
    emit("NEXT4 SwiGLU + 1x128 quant", f"gate|up [{M},{2 * F}] -> [{M},{F}]",
         lambda: _time_kernel(lambda: fb.fp8_swiglu_quant_act_1x128(gu, qa=qh, sa=sh)),
         4 * M * F + M * F + 4 * M * (F // 128), "GB/s", lambda: oracle.swiglu_quant_act_1x128(gus),
         5 * 128 * F, "rows[:128]")
    sampler.stop()
    return lines


def load_library():
    try:
        import fp8_fine_grained_14_b300 as fb

        fb.binding  # noqa: B018  (loads libfp8bs.so; raises when it is missing)
        return fb
    except ImportError:
        from fp8_fine_grained_14_b300 import build

        build.build()
        import fp8_fine_grained_14_b300 as fb

        fb.binding  # noqa: B018
        return fb


def run_ours(args):
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = init_dist(world, "nccl")
    fb = load_library()
    name = args.config
    inp = make_inputs(name, seed=rank)
    stream = torch.cuda.Stream(device)
    step = Step(name, inp, device, stream, fb)

    total_ms, per_kernel, clocks, attribution_ms, launch_mode, stamped = time_device(
        step, stream, args.steps, args.warmup, dist, device, use_graph=not args.no_graph)
    total_ms = max_over_ranks(dist, total_ms, device)
    ms_per_step = total_ms / args.steps
    flops = step.flops()
    value = flops * world / (ms_per_step * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    kern = {}
    for k, ms in per_kernel.items():
        units, bound = step.algorithmic(k)
        if bound == "tensor":
            peak = peaks["bf16_tflops"] * FP8_PER_BF16
            achieved = units / (ms * 1e-3) / 1e12
            unit = "TFLOP/s"
        else:
            peak = peaks["hbm_gbs"]
            achieved = units / (ms * 1e-3) / 1e9
            unit = "GB/s"
        kern[k] = {"us_events": ms * 1e3, "achieved_events": achieved, "unit": unit, "frac_events": achieved / peak,
                   "peak": peak, "bound": bound, "algorithmic": units}
        if stamped is not None:
            sms = stamped[0][k]
            a_st = units / (sms * 1e-3) / (1e12 if bound == "tensor" else 1e9)
            kern[k].update({"us_in_step": sms * 1e3, "achieved_in_step": a_st, "frac_in_step": a_st / peak})
        # the kernel's figure: its share of the step by device timestamps when
        # that pass ran (graph-timed steps), else its event interval
        kern[k]["us"] = kern[k].get("us_in_step", kern[k]["us_events"])
        kern[k]["frac"] = kern[k].get("frac_in_step", kern[k]["frac_events"])
    dominant = max(per_kernel, key=per_kernel.get)
    d = kern[dominant]
    roofline = {"kernel": dominant, "bound": d["bound"], "achieved": d["achieved_events"], "peak": d["peak"],
                "unit": d["unit"], "frac": d["frac_events"], "traffic": profiled_traffic(dominant, name),
                "peak_source": (f"{peak_src} " + ("bf16 burst x 2 (dense FP8/BF16 nominal ratio)"
                                                  if d["bound"] == "tensor" else "HBM copy"))}
    if d["bound"] == "tensor":
        # the same kernel against the sustained (power-capped, seconds-long)
        # cuBLAS figure; "frac" above keeps the stricter burst denominator
        sustained = peaks["bf16_tflops_sustained"] * FP8_PER_BF16
        roofline["peak_sustained"] = sustained
        roofline["frac_of_sustained"] = d["achieved_events"] / sustained
    nominal = NOMINAL["fp8_tflops"] if d["bound"] == "tensor" else NOMINAL["hbm_gbs"]
    roofline["peak_nominal"] = nominal
    roofline["frac_of_nominal"] = d["achieved_events"] / nominal
    if "frac_in_step" in d:
        roofline["achieved_in_step"] = d["achieved_in_step"]
        roofline["frac_in_step"] = d["frac_in_step"]
    for k, v in kern.items():
        v["frac_of_nominal"] = v["achieved_events"] / (NOMINAL["fp8_tflops"] if v["bound"] == "tensor"
                                                       else NOMINAL["hbm_gbs"])

    e2e = None
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 20))
        ms, wall, h2d, d2h, mode = time_e2e(name, inp, step, stream, e2e_steps, 2, device, fb)
        ms = max_over_ranks(dist, ms, device)
        e2e = {"value": flops * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": e2e_steps, "path": mode}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(name, inp)

    if rank == 0:
        M, N, K = step.M, step.N, step.K
        line = {
            "metric": "block-scaled FP8 GEMM TFLOPS (incl. quant) vs FP8 peak; quant GB/s vs HBM",
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 (f32 accumulate, bf16 out)", "data": "synthetic",
            "config": arm_config(name, M, N, K, step.G, step.kernels, world),
            "roofline": roofline,
            "kernels": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items()}
                        for k, v in kern.items()},
            "tflops_gemm_only": flops / (kern[step.kernels[-1]]["us"] * 1e-6) / 1e12,
            "timing": {"timed_region": f"{args.steps} steps, {launch_mode}, CUDA events on the launching stream",
                       "kernels_events": f"us_events: a second pass of {args.steps} stream-launched steps with a "
                                         "CUDA event after each kernel; a kernel's time includes the full launch "
                                         "gap (3-6 us) that the event record puts before it",
                       "kernels_in_step": f"us_in_step: a third pass, the {args.steps} steps as a CUDA graph with "
                                          "a device-timestamp kernel after each kernel; a kernel's time runs from "
                                          "the previous kernel's end to its own, as in the timed graph, plus "
                                          "about one short launch for the timestamp",
                       "kernels_us_frac": "us and frac: us_in_step and frac_in_step when the timestamp pass ran, "
                                          "else us_events and frac_events; the roofline object keeps the event "
                                          "figure as frac and adds frac_in_step",
                       "attribution_pass_ms_per_step": attribution_ms,
                       "stamp_pass_ms_per_step": stamped[1] if stamped is not None else None,
                       "stamp_pass_clocks": ({k: stamped[2].get(k) for k in ("sm_mhz", "reasons", "samples")}
                                             if stamped is not None else None)},
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": step_launches(step, torch.cuda.get_device_properties(device).multi_processor_count)
                            * args.steps,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="up", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time stream launches instead of a CUDA graph of the step's calls")
    ap.add_argument("--rows", action="store_true",
                    help="time every scope-table kernel on its own (one JSON line per row) and exit")
    ap.add_argument("--only", default="",
                    help="with --rows: time only the rows whose name or workload contains this text "
                         "(alternatives separated by '|')")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps; the number is not a valid measurement", file=sys.stderr)
    if args.rows:
        run_rows(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
