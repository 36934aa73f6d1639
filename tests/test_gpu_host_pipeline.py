"""The end-to-end API (HostPipeline): batches in pinned host memory, copied
in, quantised, multiplied and copied out on three overlapped streams.  Y must
equal the device-resident path bit for bit (the same kernels on the same
inputs), whether each buffer set's kernels replay from a captured CUDA graph
or are called directly, and must meet the GEMM tolerance against the oracle.
Method: "The Definitive Information To Deepseek", "Figure 7 (a)" (1x128 /
128x128 grouping) and paragraph 4 (FP8 GEMM, BF16 output)."""
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
import oracle
from fp8_fine_grained_14_b300 import workloads
from helpers import assert_gemm_close, f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(pipe, xs, ws, N):
    ys = [torch.empty((x.shape[0], N), dtype=torch.bfloat16).pin_memory() for x in xs]
    for x, w, y in zip(xs, ws, ys):
        pipe.submit(x, w, y)
    pipe.synchronize()
    return ys


@pytest.mark.parametrize("M,N,K", [(256, 512, 384), (64, 2560, 1024), (300, 256, 256)])
def test_host_pipeline_matches_device_path(M, N, K):
    batches = [workloads.dense_inputs(M, N, K, seed=40 + i) for i in range(3)]
    xs = [x.pin_memory() for x, _ in batches]
    ws = [w.pin_memory() for _, w in batches]
    pipes = [fb.HostPipeline(M, N, K, device=DEV, depth=2, use_graph=g) for g in (True, False)]
    assert pipes[0].graphed and not pipes[1].graphed
    ys_graph = _run(pipes[0], xs, ws, N)
    ys_direct = _run(pipes[1], xs, ws, N)
    assert fb.fp8bs_last_device_error() == 0
    for (x, w), yg, yd in zip(batches, ys_graph, ys_direct):
        y_dev, _ = fb.linear_forward(x.to(DEV), w.to(DEV))
        torch.cuda.synchronize()
        assert torch.equal(yg, yd) and torch.equal(yg, y_dev.cpu())
        y_ref, _ = oracle.linear_forward(f32(x), f32(w))
        assert_gemm_close(f32(yg), y_ref)


def test_host_pipeline_prequantised_weights():
    """Decode-style serving: W quantised once on the device, only X moves."""
    M, N, K = 64, 1024, 512
    _, w = workloads.dense_inputs(1, N, K, seed=7)
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    xs = [workloads.dense_inputs(M, 128, K, seed=50 + i)[0].pin_memory() for i in range(4)]
    pipe = fb.HostPipeline(M, N, K, device=DEV, depth=2, prequantised_w=(qw, sw))
    assert pipe.graphed
    ys = _run(pipe, xs, [None] * len(xs), N)
    for x, y in zip(xs, ys):
        qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
        y_dev = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
        torch.cuda.synchronize()
        assert torch.equal(y, y_dev.cpu())
