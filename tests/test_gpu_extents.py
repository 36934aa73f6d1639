"""Extents beyond one grid dimension: the kernels whose second grid
dimension is capped at 65535 walk the rest in a grid-stride loop, and the
GEMM's promotion runs over very long K.  Inputs are drawn on the device
(seeded); sampled outputs, which the oracle computes group by group, are
compared bit for bit (codes, scales, layouts) or within the GEMM tolerance.
"""
import numpy as np
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
import oracle
from helpers import assert_codes_equal, assert_gemm_close, assert_scales_equal, f32, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"
CAP = 65535


def _bf16(shape, seed, std=1.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return (torch.randn(shape, generator=g, device=DEV) * std).to(torch.bfloat16)


def test_act_quant_beyond_grid_cap():
    """M = 32 * 65535 + 100 rows: the row tiles past the grid's y extent."""
    M, K = 32 * CAP + 100, 256
    x = _bf16((M, K), 1)
    qa, sa = fb.fp8_quant_act_1x128(x)
    torch.cuda.synchronize()
    rows = np.concatenate([np.arange(64), np.arange(32 * CAP - 64, M)])
    q_ref, s_ref = oracle.quant_act_1x128(f32(x[torch.as_tensor(rows, device=DEV)]))
    assert_codes_equal(u8(qa[torch.as_tensor(rows, device=DEV)]), q_ref, "codes")
    assert_scales_equal(f32(sa)[:, rows], s_ref, "scales")


def test_weight_quant_dequant_and_transpose_beyond_grid_cap():
    """N / 128 = 65538 row blocks for the weight quantiser and 2 * 65535 + 4
    for the dequantiser (which takes blocks in pairs); K / 128 = 65537 column
    blocks for the transpose."""
    N, K = 128 * (2 * CAP + 4), 128
    w = _bf16((N, K), 2, std=0.02)
    qw, sw = fb.fp8_quant_weight_128x128(w)
    y = fb.fp8_dequant_weight_128x128(qw, sw)
    torch.cuda.synchronize()
    blocks = [0, 1, CAP - 1, CAP, CAP + 1, 2 * CAP - 1, 2 * CAP, 2 * CAP + 3]
    rows = np.concatenate([np.arange(b * 128, b * 128 + 128) for b in blocks])
    ri = torch.as_tensor(rows, device=DEV)
    q_ref, s_ref = oracle.quant_weight_128x128(f32(w[ri]))
    assert_codes_equal(u8(qw[ri]), q_ref, "codes")
    assert_scales_equal(f32(sw)[blocks], s_ref, "scales")
    y_ref = oracle.dequant_weight_128x128_bf16(q_ref, s_ref)
    assert np.array_equal(f32(y[ri]).view(np.uint32), y_ref.view(np.uint32))
    del y, w
    # transpose: W [128, 128 * (CAP + 2)] -> W^T, the K blocks past the cap
    Kt = 128 * (CAP + 2)
    g = torch.Generator(device=DEV).manual_seed(3)
    q = torch.randint(0, 256, (128, Kt), generator=g, device=DEV, dtype=torch.int32).to(torch.uint8)
    s = torch.rand((1, Kt // 128), generator=g, device=DEV)
    qt, st = fb.fp8_transpose_weight_128x128(q, s)
    torch.cuda.synchronize()
    for kb in (0, CAP - 1, CAP, CAP + 1):
        cols = slice(kb * 128, kb * 128 + 128)
        assert torch.equal(qt[cols], q[:, cols].t())
        assert st[kb, 0].item() == s[0, kb].item()


def test_swiglu_quant_beyond_grid_cap():
    """M = 32 * 65535 + 40 rows of [gate | up] with F = 128: codes and scales of
    the sampled rows equal the oracle's quantisation of the kernel's own h."""
    M, F = 32 * CAP + 40, 128
    gu = _bf16((M, 2 * F), 4)
    qa, sa, h = fb.fp8_swiglu_quant_act_1x128(gu, return_h=True)
    torch.cuda.synchronize()
    rows = np.concatenate([np.arange(32), np.arange(32 * CAP - 32, M)])
    ri = torch.as_tensor(rows, device=DEV)
    q_ref, s_ref = oracle.quant_act_1x128(f32(h[ri]))
    assert_codes_equal(u8(qa[ri]), q_ref, "codes")
    assert_scales_equal(f32(sa)[:, rows], s_ref, "scales")
    hr, _, _ = oracle.swiglu_quant_act_1x128(f32(gu[ri]))
    assert np.all(np.abs(f32(h[ri]).astype(np.float64) - hr) <= np.abs(hr) * 2.0 ** -7 + 1e-30)


def test_per_channel_beyond_grid_cap():
    """M = 64 * 65535 + 64 rows (the two-pass path, row tiles past the cap),
    16 channels: every column's scale and the codes of sampled rows."""
    M, K = 64 * CAP + 64, 16
    x = _bf16((M, K), 5)
    q, s = fb.fp8_quant_per_channel(x)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_per_channel(f32(x))
    assert_scales_equal(f32(s), s_ref, "scales")
    rows = np.concatenate([np.arange(64), np.arange(64 * CAP - 64, M)])
    assert_codes_equal(u8(q)[rows], q_ref[rows], "codes")


def test_gemm_long_k():
    """K = 131072 (1024 promotions) on a skinny grid that the launcher splits
    along K: within the tolerance of the oracle."""
    M, N, K = 64, 256, 131072
    x = _bf16((M, K), 6)
    w = _bf16((N, K), 7, std=0.02)
    qa, sa = fb.fp8_quant_act_1x128(x)
    qw, sw = fb.fp8_quant_weight_128x128(w)
    y = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    y32 = fb.fp8_blockscaled_gemm(qa, sa, qw, sw, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    y_ref = oracle.blockscaled_gemm(u8(qa), f32(sa)[:, :M], u8(qw), f32(sw))
    assert_gemm_close(f32(y32), y_ref)
    assert np.array_equal(oracle.bf16_round(f32(y32)).view(np.uint32), f32(y).view(np.uint32))
