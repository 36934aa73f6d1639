"""Packed weight tiles for weight-streaming GEMMs.

fp8_pack_weight_128x128 reorders the codes of fp8_quant_weight_128x128 into
one contiguous 16 KB image per 128x128 block ("Figure 7 (a)" item (2)
grouping; 128-byte swizzle, K-major); fp8_blockscaled_gemm_packed reads B
from it.  The layout is checked byte for byte against its definition; the
GEMM against the row-major path (bit for bit where both pick the same tile
shape) and against the oracle within |y - y_ref| <= 1e-2 |y_ref| + 1e-3 rms.
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


def _packed_reference(q):
    """The packed layout written out from its definition, with numpy indexing."""
    N, K = q.shape
    r = np.arange(128)[:, None]
    c = np.arange(128)[None, :]
    pos = 128 * r + 16 * ((c // 16) ^ (r % 8)) + (c % 16)      # [128, 128] byte positions
    out = np.zeros((N // 128, K // 128, 128 * 128), dtype=np.uint8)
    for nb in range(N // 128):
        for kb in range(K // 128):
            out[nb, kb, pos.ravel()] = q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128].ravel()
    return out


@pytest.mark.parametrize("N,K,pad", [(128, 128, 0), (384, 512, 128), (1024, 896, 16)])
def test_pack_layout(N, K, pad):
    rng = np.random.default_rng(N + K)
    q = rng.integers(0, 256, (N, K + pad)).astype(np.uint8)
    qd = torch.from_numpy(q).to(DEV)[:, :K]
    wp = fb.fp8_pack_weight_128x128(qd)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    assert np.array_equal(u8(wp), _packed_reference(q[:, :K]))


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (37, 384, 256), (64, 1024, 1024), (100, 384, 640), (300, 512, 640)])
def test_packed_gemm_bit_identical_narrow(M, N, K):
    """Skinny grids take the same single-CTA tile shape on both paths, so Y
    agrees bit for bit; and with the oracle."""
    x, w = workloads.dense_inputs(M, N, K, seed=M + 7 * N + K)
    qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    wp = fb.fp8_pack_weight_128x128(qw)
    y = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    yp = fb.fp8_blockscaled_gemm_packed(qa, sa, wp, sw)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    assert torch.equal(y, yp)
    y_ref, _ = oracle.linear_forward(f32(x), f32(w))
    assert_gemm_close(f32(yp), y_ref)


def test_packed_gemm_decode_full_size():
    """The decode workload 64 x 18432 x 7168, whole output: bit for bit the
    row-major path; sampled columns against the oracle."""
    x, w = workloads.config_inputs("decode")
    qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    wp = fb.fp8_pack_weight_128x128(qw)
    y = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    yp = fb.fp8_blockscaled_gemm_packed(qa, sa, wp, sw)
    torch.cuda.synchronize()
    assert torch.equal(y, yp)
    rows = np.arange(x.shape[0])
    blocks = sample_blocks(w.shape[0] // 128, 6, seed=3)
    _, _, _, _, y_ref, cols = oracle_dense_sampled(x, w, rows, blocks)
    assert_gemm_close(f32(yp[:, torch.as_tensor(cols, device=DEV)]), y_ref)


@pytest.mark.parametrize("M,N,K", [(1300, 4096, 384), (2048, 2560, 6144)])
def test_packed_gemm_wide(M, N, K):
    """Grids that fill the GPU run 128 x 256 single-CTA tiles on the packed
    path (CTA pairs on the row-major one), including a split-K tail: within
    the tolerance of the oracle on every row of sampled column blocks."""
    x, w = workloads.dense_inputs(M, N, K, seed=M + N)
    qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    wp = fb.fp8_pack_weight_128x128(qw)
    yp = fb.fp8_blockscaled_gemm_packed(qa, sa, wp, sw)
    yp2 = fb.fp8_blockscaled_gemm_packed(qa, sa, wp, sw)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    assert torch.equal(yp, yp2)
    rows = np.arange(M)
    blocks = [0, 3, N // 128 - 2, N // 128 - 1]
    _, _, _, _, y_ref, cols = oracle_dense_sampled(x, w, rows, blocks)
    assert_gemm_close(f32(yp[:, torch.as_tensor(cols, device=DEV)]), y_ref)
