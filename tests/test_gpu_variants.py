"""Parity of the quantisation variants with the CPU oracle: FP8 per token and
per channel, the E5M6 activation format, and SwiGLU fused with the 1x128
quantiser (the TileKernels release, "DeepSeek starts updating frequently",
item "Quantification"; E5M6 in "The Definitive Information To Deepseek",
paragraph 3).  Codes and scales bit-exact; the SwiGLU product, computed in
FP32 with the CUDA exponential, within its rounding bound of the exact
float64 value, its codes bit-exact given that product, and bit-exact with
the oracle's own end-to-end codes and scales wherever the two products
agree."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
import oracle
from fp8_fine_grained_14_b300 import workloads
from helpers import assert_codes_equal, assert_scales_equal, f32, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _edge_matrix(M, K, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= (2.0 ** rng.integers(-30, 30, size=(M, 1))).astype(np.float32)
    if M > 4:
        x[1] = 0.0
        x[2] *= 2.0 ** -110
        x[3, : K // 2] = -(2.0 ** -40)
    if K > 4:
        x[:, 1] = 0.0
        x[:, 2] *= 2.0 ** 90
    return torch.from_numpy(x).to(torch.bfloat16)


@pytest.mark.parametrize("M,K", [(1, 16), (3, 144), (130, 7168), (64, 18432), (5, 32768)])
def test_per_token(M, K):
    x = _edge_matrix(M, K, seed=M + K)
    q, s = fb.fp8_quant_per_token(x.to(DEV))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_per_token(f32(x))
    assert_codes_equal(u8(q), q_ref, "per-token codes")
    assert_scales_equal(f32(s), s_ref, "per-token scales")


@pytest.mark.parametrize("M,K", [(1, 16), (130, 144), (300, 2048), (257, 528), (2048, 144), (2049, 16),
                                 (3000, 144), (2500, 1552), (4096, 64), (4096, 7168), (4097, 144), (6000, 256)])
def test_per_channel(M, K):
    """The cluster kernel (8 CTAs share a 64-channel strip's rows): ragged
    row ranges, CTAs with no rows (M < 8 x 16), a single and a ragged last
    64-channel group, and inputs taller than 4096 rows."""
    x = _edge_matrix(M, K, seed=3 * M + K)
    q, s = fb.fp8_quant_per_channel(x.to(DEV))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_per_channel(f32(x))
    assert_codes_equal(u8(q), q_ref, "per-channel codes")
    assert_scales_equal(f32(s), s_ref, "per-channel scales")
    # repeated calls start from fresh maxima
    q2, s2 = fb.fp8_quant_per_channel(x.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(q2, q) and torch.equal(s2, s)


def test_e5m6_every_bf16_value():
    """Every finite BF16 value encoded; every finite code decoded."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    v = (bits << 16).view(np.float32)
    v = v[np.isfinite(v)]
    v = np.concatenate([v, np.zeros(8 - len(v) % 8, dtype=np.float32)])
    x = torch.from_numpy(v).to(torch.bfloat16)
    codes = fb.e5m6_encode(x.to(DEV))
    torch.cuda.synchronize()
    want = oracle.e5m6_encode_rne_satfinite(v)
    got = codes.cpu().numpy().view(np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (bad.size, v[bad[:4]], got[bad[:4]], want[bad[:4]])
    finite = np.array([c for c in range(4096) if ((c >> 6) & 0x1F) != 31], dtype=np.uint16)
    finite = np.concatenate([finite, np.zeros(8 - len(finite) % 8, dtype=np.uint16)])
    y = fb.e5m6_decode(torch.from_numpy(finite.view(np.int16)).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(f32(y).astype(np.float64), oracle.e5m6_decode(finite))


@pytest.mark.parametrize("M,F", [(1, 128), (130, 256), (33, 384), (1000, 2048), (4096, 2048)])
def test_swiglu_quant(M, F):
    g = torch.Generator().manual_seed(M + F)
    gate = torch.randn(M, F, generator=g) * 3.0
    up = torch.randn(M, F, generator=g)
    # zeros, huge |g| (exp(-g) overflows float32 for g < -88.7), results near
    # the bottom of the normal float32 range
    gate[0, :12] = torch.tensor([0.0, -120.0, 95.0, -0.0, -87.5, -88.5, 88.0, 60.0, -60.0, -30.0, 30.0, -1e-30])
    gu = torch.cat([gate, up], dim=1).to(torch.bfloat16)
    qa, sa, h = fb.fp8_swiglu_quant_act_1x128(gu.to(DEV), return_h=True)
    qa2, sa2 = fb.fp8_swiglu_quant_act_1x128(gu.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(qa, qa2) and torch.equal(sa[:, :M], sa2[:, :M])
    hg = f32(h)
    # the codes are the exact 1x128 quantisation of the BF16 product
    q_ref, s_ref = oracle.quant_act_1x128(hg)
    assert_codes_equal(u8(qa), q_ref, "swiglu codes")
    assert_scales_equal(f32(sa)[:, :M], s_ref, "swiglu scales")
    # the product: BF16 rounding of a float32 value within a few ulps of silu(g) * u
    guf = f32(gu)
    h64 = oracle.silu_mul(guf[:, :F], guf[:, F:])
    h_or, q_or, s_or = oracle.swiglu_quant_act_1x128(guf)
    h_ref = oracle.bf16_round(h64.astype(np.float32))
    assert np.array_equal(h_or.view(np.uint32), h_ref.view(np.uint32))
    differ = hg != h_ref
    assert differ.mean() < 1e-3, differ.mean()
    # end to end against the oracle's own codes and scales: every 1x128 group
    # whose 128 products agree with the oracle's bit for bit has the oracle's
    # codes and scale; in a group with a differing product, the scale is the
    # oracle's unless the group's largest magnitude differs, and where the
    # scale agrees every code of an agreeing product agrees too
    KB = F // 128
    same_h = (hg.view(np.uint32) == h_or.view(np.uint32)).reshape(M, KB, 128)
    whole = same_h.all(axis=2)
    q_gpu, q_ref = u8(qa).reshape(M, KB, 128), q_or.reshape(M, KB, 128)
    s_gpu, s_ref = f32(sa)[:, :M].T, s_or.T
    assert np.array_equal(q_gpu[whole], q_ref[whole]), "codes differ in groups whose products agree"
    assert np.array_equal(s_gpu[whole].view(np.uint32), s_ref[whole].view(np.uint32))
    amax_same = (np.max(np.abs(hg.reshape(M, KB, 128)), axis=2) ==
                 np.max(np.abs(h_or.reshape(M, KB, 128)), axis=2))
    assert np.array_equal(s_gpu[amax_same].view(np.uint32), s_ref[amax_same].view(np.uint32))
    scale_same = s_gpu.view(np.uint32) == s_ref.view(np.uint32)
    agree = same_h & scale_same[:, :, None]
    assert np.array_equal(q_gpu[agree], q_ref[agree]), "codes differ where product and scale agree"
    print(f"SwiGLU {M}x{F}: {differ.mean():.2e} of the products and {1 - whole.mean():.2e} of the 1x128 groups "
          f"differ from the oracle's (bound on products: 1e-3)")
    a = np.abs(h64[differ])
    ulp_bf16 = 2.0 ** (np.floor(np.log2(np.maximum(a, 1e-38))) - 7)
    assert np.all(np.abs(hg[differ] - h64[differ]) <= 0.5 * ulp_bf16 + a * 2.0 ** -20)
