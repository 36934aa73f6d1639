"""Parity of the backward-GEMM path with the CPU oracle.

"The Definitive Information To Deepseek": the activation is kept in FP8 for
the linear layer's backward pass (paragraph 2) and the backward is split into
its input-gradient and weight-gradient parts (paragraph 3), both FP8 GEMMs with
the "Figure 7 (a)" grouping.  dX = Q(dY) . (128x128 blocks of W, transposed);
dW = Q(dY^T) . Q(X^T)^T with 1x128 tiles of the transposes (per channel per
128 tokens) and both scales applied at each 128-token chunk's promotion.
Codes, scales and transposes bit-exact; GEMM outputs within
|y - y_ref| <= 1e-2 |y_ref| + 1e-3 rms(y_ref).
"""
import numpy as np
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
import oracle
from fp8_fine_grained_14_b300 import workloads
from helpers import assert_codes_equal, assert_gemm_close, assert_scales_equal, f32, sample_blocks, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("M,K", [(128, 128), (256, 384), (1024, 1152), (384, 7168)])
def test_quant_act_t(M, K):
    x, _ = workloads.dense_inputs(M, 128, K, seed=M + K)
    xd = x.to(DEV)
    qt, st = fb.fp8_quant_act_1x128_t(xd)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_act_1x128_t(f32(x))
    assert_codes_equal(u8(qt), q_ref, "codes of x^T")
    assert_scales_equal(f32(st)[:, :K], s_ref, "scales of x^T")
    # the same as the forward quantiser applied to x^T
    qa, sa = fb.fp8_quant_act_1x128(xd.t().contiguous())
    torch.cuda.synchronize()
    assert torch.equal(qa, qt) and torch.equal(sa[:, :K], st[:, :K])


def test_quant_act_t_edge_columns():
    """Zero columns (with -0), outlier columns, tiny (subnormal-scale) and
    huge columns, and values far below their column's resolution."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((256, 384)).astype(np.float32)
    x[:, 0] = 0.0
    x[7, 0] = -0.0
    x[:, 1] *= 100.0
    x[:, 2] *= 2.0 ** -130
    x[:, 3] *= 2.0 ** 100
    x[:, 4] = rng.standard_normal(256).astype(np.float32) * 1e4
    x[:10, 4] = -(2.0 ** -20)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    qt, st = fb.fp8_quant_act_1x128_t(xb.to(DEV))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_act_1x128_t(f32(xb))
    assert_codes_equal(u8(qt), q_ref, "codes")
    assert_scales_equal(f32(st)[:, :384], s_ref, "scales")
    assert np.all(u8(qt)[0] == 0)


@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (1024, 2048), (18432, 7168)])
def test_transpose_weight(N, K):
    _, w = workloads.dense_inputs(1, N, K, seed=N + K)
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    qwt, swt = fb.fp8_transpose_weight_128x128(qw, sw)
    torch.cuda.synchronize()
    assert torch.equal(qwt, qw.t()), "codes of W^T"
    assert torch.equal(swt, sw.t()), "scales of W^T"


def _rowscaled_case(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    a = (torch.randn(M, K, generator=g) * torch.pow(2.0, torch.randint(-6, 6, (M, 1), generator=g).float()))
    b = (torch.randn(N, K, generator=g) * torch.pow(2.0, torch.randint(-6, 6, (N, 1), generator=g).float()))
    return a.to(torch.bfloat16), b.to(torch.bfloat16)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (129, 384, 256), (300, 512, 640), (1300, 4096, 384),
                                   (64, 1024, 1024)])
def test_rowscaled_gemm(M, N, K):
    a, b = _rowscaled_case(M, N, K, seed=M + N + K)
    qa, sa = fb.fp8_quant_act_1x128(a.to(DEV))
    qb, sb = fb.fp8_quant_act_1x128(b.to(DEV))
    y16 = fb.fp8_blockscaled_gemm_rowscaled(qa, sa, qb, sb)
    y32 = fb.fp8_blockscaled_gemm_rowscaled(qa, sa, qb, sb, out_dtype=torch.float32)
    torch.cuda.synchronize()
    qa_r, sa_r = oracle.quant_act_1x128(f32(a))
    qb_r, sb_r = oracle.quant_act_1x128(f32(b))
    y_ref = oracle.blockscaled_gemm_rowscaled(qa_r, sa_r, qb_r, sb_r)
    assert_gemm_close(f32(y16), y_ref, what="bf16")
    assert_gemm_close(f32(y32), y_ref, what="f32")
    assert np.array_equal(oracle.bf16_round(f32(y32)).view(np.uint32), f32(y16).view(np.uint32))
    assert fb.fp8bs_last_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (1024, 2048, 1024)])
def test_linear_backward(M, N, K):
    x, w, dy = workloads.backward_inputs(M, N, K, seed=M + N)
    dx, dw = fb.linear_backward(x.to(DEV), w.to(DEV), dy.to(DEV))
    torch.cuda.synchronize()
    dx_ref, dw_ref = oracle.linear_backward(f32(x), f32(w), f32(dy))
    assert dx.shape == (M, K) and dw.shape == (N, K) and dw.dtype == torch.float32
    assert_gemm_close(f32(dx), dx_ref, what="dX")
    assert_gemm_close(f32(dw), dw_ref, what="dW")
    assert fb.fp8bs_last_device_error() == 0


def test_wgrad_full_size_sampled():
    """The up-projection's weight gradient dW [18432, 7168] = dY^T X over 4096
    tokens, in one launch; sampled rows of dW against the oracle (the groups of
    dY^T are per column of dY, so a column sample is exact)."""
    M, N, K = 4096, 18432, 7168
    x, _, dy = workloads.backward_inputs(M, 128, K, seed=5)  # W unused
    g = torch.Generator().manual_seed(6)
    dy = torch.randn(M, N, generator=g).to(torch.bfloat16)
    qdyt, sdyt = fb.fp8_quant_act_1x128_t(dy.to(DEV))
    qxt, sxt = fb.fp8_quant_act_1x128_t(x.to(DEV))
    dw = fb.fp8_blockscaled_gemm_rowscaled(qdyt, sdyt, qxt, sxt, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    rows = np.array(sorted(set([0, N - 1]) | set(np.random.default_rng(7).choice(N, 40, replace=False).tolist())))
    qa_r, sa_r = oracle.quant_act_1x128_t(f32(dy)[:, rows])
    qb_r, sb_r = oracle.quant_act_1x128_t(f32(x))
    assert_codes_equal(u8(qdyt)[rows], qa_r, "codes of dY^T")
    assert_scales_equal(f32(sdyt)[:, rows], sa_r, "scales of dY^T")
    assert_codes_equal(u8(qxt), qb_r, "codes of X^T")
    y_ref = oracle.blockscaled_gemm_rowscaled(qa_r, sa_r, qb_r, sb_r)
    assert_gemm_close(f32(dw)[rows], y_ref, what="dW rows")


def test_rowscaled_split_tail():
    """The row-scaled GEMM with a split-K tail (80 pair tiles on 74 resident
    pairs): every row, the last column tiles, and BF16 == RNE(FP32)."""
    M, N, K = 2048, 2560, 6144
    a, b = _rowscaled_case(M, N, K, seed=7)
    qa, sa = fb.fp8_quant_act_1x128(a.to(DEV))
    qb, sb = fb.fp8_quant_act_1x128(b.to(DEV))
    y16 = fb.fp8_blockscaled_gemm_rowscaled(qa, sa, qb, sb)
    y32 = fb.fp8_blockscaled_gemm_rowscaled(qa, sa, qb, sb, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    cols = np.arange(N - 512, N)
    qa_r, sa_r = oracle.quant_act_1x128(f32(a))
    qb_r, sb_r = oracle.quant_act_1x128(f32(b)[cols])
    y_ref = oracle.blockscaled_gemm_rowscaled(qa_r, sa_r, qb_r, sb_r)
    assert_gemm_close(f32(y32)[:, cols], y_ref, what="f32")
    assert np.array_equal(oracle.bf16_round(f32(y32)).view(np.uint32), f32(y16).view(np.uint32))
