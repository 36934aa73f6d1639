"""Bit-exact parity of the CUDA 128x128 block dequantisation (FP8 -> BF16)
with the CPU oracle: y = bf16(fl32(dec(q) * s)), the FP8-to-BF16 weight
conversion of the DeepSeek-V3 model card (section 6, "How to Run Locally"),
the inverse of the 128x128 weight quantisation of "The Definitive Information
To Deepseek" ("Figure 7 (a)" item (2))."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
import oracle
from fp8_fine_grained_14_b300 import workloads
from helpers import f32, sample_blocks, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _assert_bf16_equal(got, want, what):
    got = np.ascontiguousarray(got, dtype=np.float32)
    want = np.ascontiguousarray(want, dtype=np.float32)
    assert got.shape == want.shape
    bad = np.argwhere(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, (f"{what}: {len(bad)} values differ, first at {bad[:4].tolist()}: "
                           f"gpu={[float(got[tuple(b)]) for b in bad[:4]]} "
                           f"oracle={[float(want[tuple(b)]) for b in bad[:4]]}")


@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (1024, 1152)])
def test_dequant_of_quantised_weights(N, K):
    _, w = workloads.dense_inputs(1, N, K, seed=N + 3 * K)
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    y = fb.fp8_dequant_weight_128x128(qw, sw)
    torch.cuda.synchronize()
    _assert_bf16_equal(f32(y), oracle.dequant_weight_128x128_bf16(u8(qw), f32(sw)), "dequant")


def test_dequant_every_code_and_extreme_scales():
    """All 254 finite codes in every block; scales from subnormal to large,
    including ones whose products overflow BF16's range of exactness."""
    NB, KB = 6, 4
    rng = np.random.default_rng(5)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    q = rng.choice(finite, size=(NB * 128, KB * 128)).astype(np.uint8)
    q[:254, 0] = finite  # every code at least once
    s = np.array([[1.0, 3e-39, 0.0, 1.2345678], [2.0 ** -100, 7.77e30, 0.5, 1e-3],
                  [448.0, 1.0 / 448.0, 2.0 ** 20, 0.0078125], [1.1, 0.9, 1.5, 2.5],
                  [1e-40, 1e-20, 1e20, 3.0e35], [0.333, 0.666, 0.999, 1.001]], dtype=np.float32)
    qd = torch.from_numpy(q).to(DEV)
    sd = torch.from_numpy(s).to(DEV)
    y = fb.fp8_dequant_weight_128x128(qd, sd)
    torch.cuda.synchronize()
    _assert_bf16_equal(f32(y), oracle.dequant_weight_128x128_bf16(q, s), "dequant")


def test_dequant_expert_stack_and_strides():
    G, N, K = 3, 256, 384
    _, w = workloads.dense_inputs(1, G * N, K, seed=99)
    qw, sw = fb.fp8_quant_weight_128x128(w.reshape(G, N, K).to(DEV))
    y = fb.fp8_dequant_weight_128x128(qw, sw)
    ref = oracle.dequant_weight_128x128_bf16(u8(qw).reshape(G * N, K), f32(sw).reshape(G * N // 128, K // 128))
    torch.cuda.synchronize()
    _assert_bf16_equal(f32(y).reshape(G * N, K), ref, "stack")
    # strided codes and output, guard columns untouched
    qbig = torch.zeros((N, K + 128), dtype=torch.uint8, device=DEV)
    qbig[:, :K] = qw[0]
    ybig = torch.full((N, K + 64), 5.0, dtype=torch.bfloat16, device=DEV)
    fb.fp8_dequant_weight_128x128(qbig[:, :K], sw[0].contiguous(), y=ybig[:, :K])
    torch.cuda.synchronize()
    _assert_bf16_equal(f32(ybig)[:, :K], ref[:N], "strided")
    assert torch.all(ybig[:, K:] == 5.0)


def test_dequant_full_size_sampled():
    """The up-projection weight [18432, 7168] in one launch; sampled 128-row
    block rows compared bit for bit."""
    _, w = workloads.config_inputs("up")
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    y = fb.fp8_dequant_weight_128x128(qw, sw)
    torch.cuda.synchronize()
    blocks = sample_blocks(w.shape[0] // 128, 6, seed=8)
    rows = np.concatenate([np.arange(b * 128, b * 128 + 128) for b in blocks])
    ref = oracle.dequant_weight_128x128_bf16(u8(qw)[rows], f32(sw)[blocks])
    _assert_bf16_equal(f32(y)[rows], ref, "up weights")
