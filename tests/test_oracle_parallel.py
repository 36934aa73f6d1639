"""The row-parallel oracle runner (oracle.parallel) returns exactly what the
serial oracle returns on the whole arrays: slicing is exact because 1x128
groups lie in one row, 128x128 blocks in one 128-row slab, and an output row
of the GEMM depends only on its own row ("The Definitive Information To
Deepseek", paragraph 3, "Figure 7 (a)").  CPU only."""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_14_b300 import workloads
from helpers import bf16_bits, f32
from oracle.parallel import OraclePool, _slices


@pytest.fixture(scope="module")
def pool():
    with OraclePool(workers=3) as p:
        yield p


def test_slices_cover_and_align():
    for n, parts, align in [(1, 4, 1), (1000, 7, 1), (1024, 5, 128), (130, 12, 128), (5, 10, 1)]:
        s = _slices(n, parts, align)
        assert s[0][0] == 0 and s[-1][1] == n
        assert all(a < b for a, b in s)
        assert all(s[i][1] == s[i + 1][0] for i in range(len(s) - 1))
        assert all(a % align == 0 for a, _ in s)


def test_dense_equals_serial(pool):
    x, w = workloads.dense_inputs(333, 384, 640, seed=5, outlier_frac=0.01, outlier_scale=100.0)
    qa, sa = pool.quant_act_1x128(bf16_bits(x))
    qw, sw = pool.quant_weight_128x128(bf16_bits(w))
    y = pool.blockscaled_gemm(qa, sa, qw, sw)
    y_ref, (qa_r, sa_r, qw_r, sw_r) = oracle.linear_forward(f32(x), f32(w))
    assert np.array_equal(qa, qa_r) and np.array_equal(qw, qw_r)
    assert np.array_equal(sa.view(np.uint32), sa_r.view(np.uint32))
    assert np.array_equal(sw.view(np.uint32), sw_r.view(np.uint32))
    assert np.array_equal(y.view(np.uint64), y_ref.view(np.uint64))
    # float32 inputs give the same as BF16 bit patterns
    qa2, sa2 = pool.quant_act_1x128(f32(x))
    assert np.array_equal(qa2, qa) and np.array_equal(sa2, sa)


def test_grouped_equals_serial(pool):
    counts = [3, 0, 200, 1, 77, 0]
    G, N, K = len(counts), 256, 384
    offsets = workloads.grouped_offsets(counts)
    x, _ = workloads.dense_inputs(int(offsets[-1]), 128, K, seed=8)
    _, w = workloads.dense_inputs(1, G * N, K, seed=9)
    qa, sa = oracle.quant_act_1x128(f32(x))
    qw, sw = oracle.quant_weight_128x128(f32(w))
    qw, sw = qw.reshape(G, N, K), sw.reshape(G, N // 128, K // 128)
    y = pool.blockscaled_grouped_gemm(offsets.numpy(), qa, sa, qw, sw)
    y_ref = oracle.blockscaled_grouped_gemm(offsets.numpy(), qa, sa, qw, sw)
    assert np.array_equal(y.view(np.uint64), y_ref.view(np.uint64))


def test_bf16_bits_roundtrip():
    t = torch.randn(7, 9).to(torch.bfloat16)
    b = bf16_bits(t)
    assert b.dtype == np.int16
    assert np.array_equal((b.view(np.uint16).astype(np.uint32) << 16).view(np.float32), f32(t))
