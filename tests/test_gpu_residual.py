"""Parity of the block-scaled GEMM with a fused BF16 residual add.

Y = bf16_rn(fl32(sum of the promoted K chunks) + R): the FP32 result of the
GEMM ("The Definitive Information To Deepseek", paragraphs 1 and 4; outputs
in BF16 or FP32) and the residual stream R are added in FP32 and rounded once.
Two checks per case:

- against the oracle (float64 GEMM + R) within the GEMM tolerance
  |y_gpu - y_ref| <= 1e-2 |y_ref| + 1e-3 rms(y_ref);
- bit for bit against the FP32-output GEMM of the same operands plus R, one
  float32 addition and one BF16 rounding on the host (the epilogue reads the
  same FP32 accumulator for every output format).
"""
import numpy as np
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
import oracle
from fp8_fine_grained_14_b300 import workloads
from helpers import assert_gemm_close, f32, oracle_dense_sampled, sample_blocks, sample_rows, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _residual(M, N, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((M, N), generator=g) * scale).to(torch.bfloat16)


def _operands(x, w):
    qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    return qa, sa, qw, sw


def _host_sum(y32, r):
    return oracle.bf16_round(np.float32(f32(y32)) + np.float32(f32(r)))


def _check(x, w, r, in_place=False):
    qa, sa, qw, sw = _operands(x, w)
    rd = r.to(DEV)
    y32 = fb.fp8_blockscaled_gemm(qa, sa, qw, sw, out_dtype=torch.float32)
    if in_place:
        y = rd.clone()
        out = fb.fp8_blockscaled_gemm_residual(qa, sa, qw, sw, y, y=y)
        assert out.data_ptr() == y.data_ptr()
    else:
        y = fb.fp8_blockscaled_gemm_residual(qa, sa, qw, sw, rd)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    assert torch.equal(rd.cpu(), r)  # the residual input is not written unless it is the output
    assert np.array_equal(_host_sum(y32, r).view(np.uint32), f32(y).view(np.uint32))
    return y, (qa, sa, qw, sw)


@pytest.mark.parametrize("M,N,K", [
    (1, 128, 128),
    (127, 128, 384),
    (129, 384, 256),   # ragged M tail, odd number of column blocks
    (300, 512, 640),
    (1300, 4096, 384),  # 256-wide tiles with a ragged M tail
])
def test_residual_against_oracle(M, N, K):
    x, w = workloads.dense_inputs(M, N, K, seed=M + 11 * N + K)
    r = _residual(M, N, seed=M + N)
    y, (qa, sa, qw, sw) = _check(x, w, r)
    y_ref = oracle.blockscaled_gemm_residual(u8(qa), f32(sa)[:, :M], u8(qw), f32(sw), f32(r))
    assert_gemm_close(f32(y), y_ref, what="gemm+residual")


def test_residual_in_place():
    """Y written over R (the residual stream updated in place)."""
    M, N, K = 300, 512, 640
    x, w = workloads.dense_inputs(M, N, K, seed=77)
    _check(x, w, _residual(M, N, seed=78), in_place=True)


def test_residual_strided():
    """R and Y as column slices of wider buffers, with different strides;
    the columns beyond N stay untouched."""
    M, N, K = 200, 384, 512
    x, w = workloads.dense_inputs(M, N, K, seed=79)
    qa, sa, qw, sw = _operands(x, w)
    rbig = _residual(M, N + 64, seed=80).to(DEV)
    ybig = torch.full((M, N + 128), -2.0, dtype=torch.bfloat16, device=DEV)
    fb.fp8_blockscaled_gemm_residual(qa, sa, qw, sw, rbig[:, :N], y=ybig[:, :N])
    y32 = fb.fp8_blockscaled_gemm(qa, sa, qw, sw, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.all(ybig[:, N:] == -2.0)
    assert np.array_equal(_host_sum(y32, rbig[:, :N].cpu()).view(np.uint32), f32(ybig[:, :N]).view(np.uint32))


def test_residual_cancellation():
    """R = -bf16(Y): the sum is the small rounding remainder of the GEMM's
    FP32 result, exact in FP32 and then rounded once."""
    M, N, K = 256, 256, 512
    x, w = workloads.dense_inputs(M, N, K, seed=81)
    qa, sa, qw, sw = _operands(x, w)
    y16 = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    r = (-y16).cpu()
    _check(x, w, r)


@pytest.mark.parametrize("M,N,K", [(2048, 2560, 6144), (2148, 2560, 6144)])
def test_residual_split_tail(M, N, K):
    """Shapes whose last round of tiles is split along K: the residual is
    added by the reduction kernel after the slices are summed."""
    x, w = workloads.dense_inputs(M, N, K, seed=M + 13 * N + K)
    r = _residual(M, N, seed=82, scale=0.5)
    y, _ = _check(x, w, r)
    rows = np.arange(M)
    blocks = [0, N // 128 - 2, N // 128 - 1]
    _, _, _, _, y_gemm, cols = oracle_dense_sampled(x, w, rows, blocks)
    y_ref = y_gemm + f32(r)[:, cols].astype(np.float64)
    assert_gemm_close(f32(y[:, torch.as_tensor(cols, device=DEV)]), y_ref, what="gemm+residual")


def test_residual_full_size_sampled():
    """The dense up-projection workload, sampled rows and column blocks."""
    x, w = workloads.config_inputs("up")
    M, N = x.shape[0], w.shape[0]
    r = _residual(M, N, seed=83)
    y, _ = _check(x, w, r)
    rows = sample_rows(M, 96, seed=84)
    blocks = sample_blocks(N // 128, 3, seed=85)
    _, _, _, _, y_gemm, cols = oracle_dense_sampled(x, w, rows, blocks)
    y_ref = y_gemm + f32(r)[rows][:, cols].astype(np.float64)
    sub = y[torch.as_tensor(rows, device=DEV)][:, torch.as_tensor(cols, device=DEV)]
    assert_gemm_close(f32(sub), y_ref, what="gemm+residual")
