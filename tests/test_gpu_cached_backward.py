"""Parity of the weight-gradient operand taken from the FP8-cached activation.

"The Definitive Information To Deepseek", paragraph 2: the activation is kept
in FP8 for the linear layer's backward pass.  The forward's 1x128 codes and
scales of X are dequantised to BF16 (bf16_rn(fl32(dec(q) * s))) and quantised
on 1x128 tiles of X^T (per channel per 128 tokens).  Codes and scales are
compared with the oracle bit for bit; dW within
|y - y_ref| <= 1e-2 |y_ref| + 1e-3 rms(y_ref).
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


def _requant_parity(qa, sa, M, K):
    """qa, sa on the device; checks the GPU requantisation against the oracle."""
    qt, st = fb.fp8_requant_act_1x128_t(qa, sa)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    q_ref, s_ref = oracle.requant_act_1x128_t(u8(qa)[:, :K], f32(sa)[:, :M])
    assert_codes_equal(u8(qt), q_ref, "requantised codes of x^T")
    assert_scales_equal(f32(st)[:, :K], s_ref, "requantised scales of x^T")
    return qt, st


@pytest.mark.parametrize("M,K", [(128, 128), (256, 384), (1024, 1152), (384, 7168)])
def test_requant_from_forward_cache(M, K):
    """The cache as the forward leaves it: fp8_quant_act_1x128 of BF16 X."""
    x, _ = workloads.dense_inputs(M, 128, K, seed=3 * M + K)
    qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
    torch.cuda.synchronize()
    q_fwd, s_fwd = oracle.quant_act_1x128(f32(x))
    assert_codes_equal(u8(qa), q_fwd, "forward codes")
    _requant_parity(qa, sa, M, K)


def test_requant_every_code_and_scale_range():
    """All 254 finite codes (with -0), all-zero groups with s = 0, and row
    scales from 2^-140 (products far into the subnormal range) to 2^100;
    strided codes and scales."""
    rng = np.random.default_rng(11)
    M, K = 512, 768
    q = rng.integers(0, 256, (M, K)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x80
    q[:, :254] = np.concatenate([np.arange(0, 0x7F), np.arange(0x80, 0xFF)]).astype(np.uint8)[None, :]
    e = rng.integers(-140, 100, (K // 128, M)).astype(np.float64)
    s = (np.ldexp(1.0, e.astype(int)) * rng.uniform(1.0, 2.0, e.shape)).astype(np.float32)
    s[:, 200] = 0.0
    q[200, :] = 0                       # an all-zero row: every group of it has s = 0
    s[1, 256:384] = 0.0
    q[256:384, 128:256] = 0             # a whole 128x128 tile of zeros
    qbig = torch.zeros((M, K + 128), dtype=torch.uint8)
    qbig[:, :K] = torch.from_numpy(q)
    sbig = torch.full((K // 128, M + 64), 7.0, dtype=torch.float32)
    sbig[:, :M] = torch.from_numpy(s)
    qd, sd = qbig.to(DEV), sbig.to(DEV)
    qt, st = _requant_parity(qd[:, :K], sd[:, :M + 64], M, K)
    assert np.all(u8(qt)[128:256, 256:384] == 0) and np.all(f32(st)[2, 128:256] == 0)


def test_requant_power_of_two_identity():
    """Power-of-two scales constant per 128x128 tile and a +-448 code in every
    column of every tile: the requantised codes are the cached ones
    transposed, bit for bit."""
    rng = np.random.default_rng(13)
    M, K = 384, 512
    q = rng.integers(0, 256, (M, K)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x05
    for mb in range(M // 128):
        q[mb * 128 + rng.integers(0, 128, K), np.arange(K)] = 0x7E if mb % 2 == 0 else 0xFE
    e = rng.integers(-20, 20, (K // 128, M // 128))
    sa = np.repeat(np.ldexp(1.0, e), 128, axis=1).astype(np.float32)
    qt, st = fb.fp8_requant_act_1x128_t(torch.from_numpy(q).to(DEV), torch.from_numpy(sa).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(u8(qt), q.T)
    assert np.array_equal(f32(st)[:, :K], np.repeat(np.ldexp(1.0, e.T), 128, axis=1).astype(np.float32))


def test_requant_full_size():
    """The up-projection's activation X [4096, 7168], whole."""
    x, _ = workloads.dense_inputs(4096, 128, 7168, seed=17)
    qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
    _requant_parity(qa, sa, 4096, 7168)


@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (1024, 2048, 1024)])
def test_linear_backward_from_cache(M, N, K):
    x, w, dy = workloads.backward_inputs(M, N, K, seed=M + 2 * N)
    qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
    dx, dw = fb.linear_backward(None, w.to(DEV), dy.to(DEV), x_cache=(qa, sa))
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    qa_r, sa_r = oracle.quant_act_1x128(f32(x))
    dx_ref, dw_ref = oracle.linear_backward_cached(qa_r, sa_r, f32(w), f32(dy))
    assert dw.dtype == torch.float32
    assert_gemm_close(f32(dx), dx_ref, what="dX")
    assert_gemm_close(f32(dw), dw_ref, what="dW from the FP8 cache")
