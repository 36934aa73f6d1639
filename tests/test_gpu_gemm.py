"""Parity of the CUDA block-scaled FP8 GEMM with the CPU oracle.

Y = sum over 128-wide K chunks of (sa * sw) * (FP8 chunk product), BF16 out
("The Definitive Information To Deepseek", paragraphs 1 and 4; scale groups
from "Figure 7 (a)").  The GPU runs the whole path (its own quantisation, then
the GEMM); the oracle quantises the same BF16 inputs itself.  Codes and
scales are compared bit for bit, Y within
|y_gpu - y_ref| <= 1e-2 |y_ref| + 1e-3 rms(y_ref).
"""
import numpy as np
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
import oracle
from fp8_fine_grained_14_b300 import workloads
from helpers import (assert_codes_equal, assert_gemm_close, assert_scales_equal, f32, oracle_dense_sampled,
                     sample_blocks, sample_rows, u8)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _full_parity(x_cpu, w_cpu):
    y, (qa, sa, qw, sw) = fb.linear_forward(x_cpu.to(DEV), w_cpu.to(DEV))
    torch.cuda.synchronize()
    y_ref, (qa_r, sa_r, qw_r, sw_r) = oracle.linear_forward(f32(x_cpu), f32(w_cpu))
    M = x_cpu.shape[0]
    assert_codes_equal(u8(qa), qa_r, "qa")
    assert_scales_equal(f32(sa)[:, :M], sa_r, "sa")
    assert_codes_equal(u8(qw), qw_r, "qw")
    assert_scales_equal(f32(sw), sw_r, "sw")
    assert_gemm_close(f32(y), y_ref)
    assert fb.fp8bs_last_device_error() == 0
    return y, y_ref


def test_tiny_config():
    x, w = workloads.config_inputs("tiny")
    _full_parity(x, w)


@pytest.mark.parametrize("M,N,K", [
    (1, 128, 128),      # single row, single chunk
    (3, 256, 256),
    (127, 128, 384),
    (129, 384, 256),    # ragged M tail, odd number of 128-column blocks
    (300, 512, 640),    # several M and N tiles, 5 chunks
    (64, 1024, 1024),   # decode-like skinny M
])
def test_narrow_tiles(M, N, K):
    x, w = workloads.dense_inputs(M, N, K, seed=M * 7 + N + K)
    _full_parity(x, w)


@pytest.mark.parametrize("M,N,K", [
    (1280, 4096, 512),  # >= one wave of 256-wide tiles
    (1300, 4096, 384),  # ragged M with 256-wide tiles
])
def test_wide_tiles(M, N, K):
    x, w = workloads.dense_inputs(M, N, K, seed=M + N + K)
    _full_parity(x, w)


def test_closed_form_constant_operands():
    """X = a, W = b everywhere: every code 0x7E, Y = K (448 s_x)(448 s_w)."""
    M, N, K = 200, 512, 768
    x = torch.full((M, K), 1.5, dtype=torch.bfloat16)
    w = torch.full((N, K), -0.0390625, dtype=torch.bfloat16)
    y, y_ref = _full_parity(x, w)
    assert np.all(y_ref == y_ref[0, 0])
    assert np.all(f32(y) == f32(y)[0, 0])


def test_outlier_channels():
    """Down-projection-like activations: a few channels x100."""
    x, w = workloads.dense_inputs(256, 384, 2048, seed=9, outlier_frac=0.01, outlier_scale=100.0)
    _full_parity(x, w)


def test_zero_groups_and_rows():
    x, w = workloads.dense_inputs(130, 256, 512, seed=11)
    x[5] = 0
    x[:, 128:256] = 0
    w[:, 384:512] = 0
    _full_parity(x, w)


def test_strided_output_and_operands():
    M, N, K = 150, 256, 384
    x, w = workloads.dense_inputs(M, N, K, seed=13)
    xd, wd = x.to(DEV), w.to(DEV)
    qa = torch.empty((M, K + 128), dtype=torch.uint8, device=DEV)[:, :K]
    sa = torch.empty((K // 128, 160), dtype=torch.float32, device=DEV)
    qw = torch.empty((N, K + 256), dtype=torch.uint8, device=DEV)[:, :K]
    fb.fp8_quant_act_1x128(xd, qa=qa, sa=sa)
    _, sw = fb.fp8_quant_weight_128x128(wd, qw=qw)
    ybig = torch.full((M, N + 64), 7.0, dtype=torch.bfloat16, device=DEV)
    fb.fp8_blockscaled_gemm(qa, sa, qw, sw, y=ybig[:, :N])
    torch.cuda.synchronize()
    y_ref, _ = oracle.linear_forward(f32(x), f32(w))
    assert_gemm_close(f32(ybig)[:, :N], y_ref)
    assert np.all(f32(ybig)[:, N:] == 7.0), "columns beyond N must be untouched"


def test_output_guard_rows():
    """Rows beyond M in a larger buffer stay untouched (ragged last tile)."""
    M, N, K = 133, 256, 256
    x, w = workloads.dense_inputs(M, N, K, seed=17)
    xd, wd = x.to(DEV), w.to(DEV)
    qa, sa = fb.fp8_quant_act_1x128(xd)
    qw, sw = fb.fp8_quant_weight_128x128(wd)
    ybuf = torch.full((M + 128, N), -3.0, dtype=torch.bfloat16, device=DEV)
    fb.fp8_blockscaled_gemm(qa, sa, qw, sw, y=ybuf[:M])
    torch.cuda.synchronize()
    assert np.all(f32(ybuf)[M:] == -3.0)
    y_ref, _ = oracle.linear_forward(f32(x), f32(w))
    assert_gemm_close(f32(ybuf)[:M], y_ref)


@pytest.mark.parametrize("M,N,K", [(129, 384, 256), (300, 512, 640), (1300, 4096, 384), (64, 1024, 1024)])
def test_f32_output(M, N, K):
    """FP32 output ("outputs in BF16 or FP32", paragraph 4): within the GEMM
    tolerance of the oracle, and the BF16 output is exactly its RNE rounding
    (both epilogues read the same FP32 accumulator)."""
    x, w = workloads.dense_inputs(M, N, K, seed=M + 5 * N + K)
    xd, wd = x.to(DEV), w.to(DEV)
    qa, sa = fb.fp8_quant_act_1x128(xd)
    qw, sw = fb.fp8_quant_weight_128x128(wd)
    y32 = fb.fp8_blockscaled_gemm(qa, sa, qw, sw, out_dtype=torch.float32)
    y16 = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    torch.cuda.synchronize()
    assert y32.dtype == torch.float32
    y_ref, _ = oracle.linear_forward(f32(x), f32(w))
    assert_gemm_close(f32(y32), y_ref)
    assert np.array_equal(oracle.bf16_round(f32(y32)).view(np.uint32), f32(y16).view(np.uint32))
    assert fb.fp8bs_last_device_error() == 0


def test_f32_output_strided_and_full_size_sampled():
    x, w = workloads.config_inputs("up")
    xd, wd = x.to(DEV), w.to(DEV)
    qa, sa = fb.fp8_quant_act_1x128(xd)
    qw, sw = fb.fp8_quant_weight_128x128(wd)
    M, N = x.shape[0], w.shape[0]
    ybig = torch.full((M, N + 32), -1.0, dtype=torch.float32, device=DEV)
    fb.fp8_blockscaled_gemm(qa, sa, qw, sw, y=ybig[:, :N])
    y16 = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    torch.cuda.synchronize()
    assert torch.all(ybig[:, N:] == -1.0)
    rows = sample_rows(M, 128, seed=31)
    blocks = sample_blocks(N // 128, 4, seed=32)
    _, _, _, _, y_ref, cols = oracle_dense_sampled(x, w, rows, blocks)
    sub = ybig[torch.as_tensor(rows, device=DEV)][:, torch.as_tensor(cols, device=DEV)]
    assert_gemm_close(f32(sub), y_ref)
    assert np.array_equal(oracle.bf16_round(f32(ybig[:, :N])).view(np.uint32), f32(y16).view(np.uint32))


@pytest.mark.parametrize("M,N,K", [(2048, 2560, 6144), (2148, 2560, 6144)])
def test_split_tail(M, N, K):
    """80 (or 90) CTA-pair tiles on 74 resident pairs leave a last round of a
    few tiles, which the launcher splits along K over the idle SMs and sums in
    a second kernel.  Every row and the last column tiles (where the tail tiles
    lie in the M-fastest order) are checked against the oracle; BF16 is the
    rounding of FP32; repeated launches give identical bits (the slices are
    summed in a fixed order)."""
    x, w = workloads.dense_inputs(M, N, K, seed=M + 3 * N + K)
    xd, wd = x.to(DEV), w.to(DEV)
    qa, sa = fb.fp8_quant_act_1x128(xd)
    qw, sw = fb.fp8_quant_weight_128x128(wd)
    y16 = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    y32 = fb.fp8_blockscaled_gemm(qa, sa, qw, sw, out_dtype=torch.float32)
    y16b = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    assert torch.equal(y16, y16b)
    assert np.array_equal(oracle.bf16_round(f32(y32)).view(np.uint32), f32(y16).view(np.uint32))
    rows = np.arange(M)
    blocks = [0, 5, N // 128 - 4, N // 128 - 3, N // 128 - 2, N // 128 - 1]
    _, _, _, _, y_ref, cols = oracle_dense_sampled(x, w, rows, blocks)
    sub = y32[:, torch.as_tensor(cols, device=DEV)]
    assert_gemm_close(f32(sub), y_ref)
