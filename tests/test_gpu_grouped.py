"""Parity of the grouped (per-expert) block-scaled GEMM with the CPU oracle.

MoE row groups: rows off[g]..off[g+1]-1 use expert g's 128x128-quantised
weights; activations are quantised per 1x128 tile over the concatenated rows
("The Definitive Information To Deepseek", "Figure 7 (a)").  Empty and
ragged groups are part of the contract.
"""
import numpy as np
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
import oracle
from fp8_fine_grained_14_b300 import workloads
from helpers import assert_codes_equal, assert_gemm_close, assert_scales_equal, f32, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _grouped_gpu(offsets, x, w):
    xd, wd = x.to(DEV), w.to(DEV)
    qa, sa = fb.fp8_quant_act_1x128(xd)
    qw, sw = fb.fp8_quant_weight_128x128(wd)
    y = fb.fp8_blockscaled_grouped_gemm(offsets.to(DEV), int(offsets[-1]), qa, sa, qw, sw)
    torch.cuda.synchronize()
    return y, qa, sa, qw, sw


@pytest.mark.parametrize("counts,N,K", [
    ([3, 0, 130, 1, 0, 257], 256, 256),
    ([128, 128], 128, 384),
    ([0, 0, 1], 384, 128),
    ([500], 512, 256),
    ([77, 300, 0, 129, 5, 64, 200, 1], 1024, 512),  # 256-wide tiles across ragged groups
    # 256-wide pair tiles: these counts put 0, 1, 127, 128, 129, 255 and 256
    # rows after a group's whole 256-row tiles (one or both CTAs of its last
    # pair masked), first and last groups included
    ([1, 256, 257, 384, 385, 128, 0, 129, 511, 640, 127, 768], 512, 384),
    ([0, 0, 300], 256, 256),
])
def test_grouped_small(counts, N, K):
    G = len(counts)
    offsets = workloads.grouped_offsets(counts)
    x, _ = workloads.dense_inputs(int(offsets[-1]), 128, K, seed=G + N)
    _, w = workloads.dense_inputs(1, G * N, K, seed=G + N + 1)
    w = w.reshape(G, N, K)
    y, qa, sa, qw, sw = _grouped_gpu(offsets, x, w)
    assert fb.fp8bs_last_device_error() == 0
    qa_r, sa_r = oracle.quant_act_1x128(f32(x))
    qw_r, sw_r = oracle.quant_weight_128x128(f32(w).reshape(G * N, K))
    assert_codes_equal(u8(qa), qa_r, "qa")
    assert_scales_equal(f32(sa)[:, : int(offsets[-1])], sa_r, "sa")
    assert_codes_equal(u8(qw).reshape(G * N, K), qw_r, "qw")
    assert_scales_equal(f32(sw).reshape(G * N // 128, K // 128), sw_r, "sw")
    y_ref = oracle.blockscaled_grouped_gemm(offsets.numpy(), qa_r, sa_r, qw_r.reshape(G, N, K),
                                            sw_r.reshape(G, N // 128, K // 128))
    assert_gemm_close(f32(y), y_ref)


def test_grouped_f32_output():
    counts = [77, 300, 0, 129, 5]
    G, N, K = len(counts), 512, 384
    offsets = workloads.grouped_offsets(counts)
    x, _ = workloads.dense_inputs(int(offsets[-1]), 128, K, seed=3)
    _, w = workloads.dense_inputs(1, G * N, K, seed=4)
    w = w.reshape(G, N, K)
    y16, qa, sa, qw, sw = _grouped_gpu(offsets, x, w)
    y32 = fb.fp8_blockscaled_grouped_gemm(offsets.to(DEV), int(offsets[-1]), qa, sa, qw, sw, out_dtype=torch.float32)
    torch.cuda.synchronize()
    qa_r, sa_r = oracle.quant_act_1x128(f32(x))
    qw_r, sw_r = oracle.quant_weight_128x128(f32(w).reshape(G * N, K))
    y_ref = oracle.blockscaled_grouped_gemm(offsets.numpy(), qa_r, sa_r, qw_r.reshape(G, N, K),
                                            sw_r.reshape(G, N // 128, K // 128))
    assert_gemm_close(f32(y32), y_ref)
    assert np.array_equal(oracle.bf16_round(f32(y32)).view(np.uint32), f32(y16).view(np.uint32))


def test_grouped_bad_offsets_reported():
    """A decreasing offset table is detected on the device and reported."""
    N, K = 128, 128
    offsets = torch.tensor([0, 100, 50, 150], dtype=torch.int32)
    x, _ = workloads.dense_inputs(150, 128, K, seed=1)
    _, w = workloads.dense_inputs(1, 3 * N, K, seed=2)
    _grouped_gpu(offsets, x, w.reshape(3, N, K))
    assert fb.fp8bs_last_device_error() == 1  # FP8BS_ERR_INVALID_ARG
    assert fb.fp8bs_last_device_error() == 0  # cleared by the read
