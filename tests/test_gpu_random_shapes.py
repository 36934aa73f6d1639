"""Parity over seeded random shapes: the forward path (1x128 activation
quantisation, 128x128 weight quantisation, the block-scaled GEMM with BF16,
FP32 and residual outputs), the grouped GEMM, both backward GEMMs (X in BF16
and from its FP8 cache), the GEMM on packed weight tiles, and the per-token
and per-channel quantisers, on shapes drawn at random rather than picked by
hand, so that tile-shape choices (64-row, 128-wide, 256-wide and CTA-pair
tiles; split and unsplit K tails; ragged M and empty groups) meet sizes
nobody chose for them.

Scale groups as in "The Definitive Information To Deepseek", "Figure 7 (a)";
the GEMM as in its paragraphs 1 and 4 (FP8 chunk products promoted with the
two scales, BF16 or FP32 out).  Codes and scales are compared bit for bit, Y
within |y_gpu - y_ref| <= 1e-2 |y_ref| + 1e-3 rms(y_ref); the BF16 and
residual outputs are also checked bit for bit against the FP32 output of the
same call (one rounding, and one FP32 addition of R before it).

Shape recipe (numpy default_rng, fixed seeds): M log-uniform within each
case's range, N and K multiples of 128, M*N*K capped so that the oracle
finishes each case in seconds; the "pair" cases take N a multiple of 256 and
enough 128-row tiles to fill the 148 SMs' worth of 256-wide tiles.  Values:
workloads.dense_inputs with a drawn weight scale and, in half the cases, a
few activation channels scaled up (down-projection-like outliers)."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
import oracle
from fp8_fine_grained_14_b300 import workloads
from helpers import assert_codes_equal, assert_gemm_close, assert_scales_equal, f32, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"
MAX_MACS = 6e9

# (kind, M range, N range in 128-blocks, K range in 128-blocks)
_KINDS = {
    "skinny": ((1, 64), (1, 64), (1, 24)),
    "narrow": ((65, 1500), (1, 24), (1, 12)),
    "pair": ((1200, 2700), (8, 20), (1, 8)),
}


def _draw_dense(kind, seed):
    rng = np.random.default_rng(seed)
    (m0, m1), (n0, n1), (k0, k1) = _KINDS[kind]
    while True:
        M = int(np.exp(rng.uniform(np.log(m0), np.log(m1 + 1))))
        M = min(max(M, m0), m1)
        nb = int(rng.integers(n0, n1 + 1))
        if kind == "pair":
            nb += nb % 2  # N a multiple of 256
        N, K = 128 * nb, 128 * int(rng.integers(k0, k1 + 1))
        if kind == "pair" and -(-M // 128) * (N // 256) < 148:
            continue
        if M * N * K <= MAX_MACS:
            break
    w_std = float(10.0 ** rng.uniform(-3, 0))
    outliers = bool(rng.integers(0, 2))
    return M, N, K, w_std, outliers


_DENSE = [(kind, 1000 + 17 * i) for i, kind in
          enumerate(["skinny"] * 5 + ["narrow"] * 5 + ["pair"] * 4)]


@pytest.mark.parametrize("kind,seed", _DENSE)
def test_random_dense(kind, seed):
    M, N, K, w_std, outliers = _draw_dense(kind, seed)
    x, w = workloads.dense_inputs(M, N, K, seed=seed, w_std=w_std,
                                  outlier_frac=0.01 if outliers else 0.0, outlier_scale=100.0)
    g = torch.Generator().manual_seed(seed + 1)
    r = (torch.randn((M, N), generator=g) * 0.5).to(torch.bfloat16)
    xd, wd, rd = x.to(DEV), w.to(DEV), r.to(DEV)
    y, (qa, sa, qw, sw) = fb.linear_forward(xd, wd)
    y32 = fb.fp8_blockscaled_gemm(qa, sa, qw, sw, out_dtype=torch.float32)
    yr = fb.fp8_blockscaled_gemm_residual(qa, sa, qw, sw, rd)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    what = f"{kind} M={M} N={N} K={K}"

    y_ref, (qa_r, sa_r, qw_r, sw_r) = oracle.linear_forward(f32(x), f32(w))
    assert_codes_equal(u8(qa), qa_r, f"qa {what}")
    assert_scales_equal(f32(sa)[:, :M], sa_r, f"sa {what}")
    assert_codes_equal(u8(qw), qw_r, f"qw {what}")
    assert_scales_equal(f32(sw), sw_r, f"sw {what}")
    assert_gemm_close(f32(y), y_ref, what=f"bf16 {what}")
    assert_gemm_close(f32(y32), y_ref, what=f"f32 {what}")
    yr_ref = oracle.blockscaled_gemm_residual(qa_r, sa_r, qw_r, sw_r, f32(r))
    assert_gemm_close(f32(yr), yr_ref, what=f"residual {what}")
    # one epilogue, one FP32 accumulator: BF16 = RNE(FP32), residual = RNE(FP32 + R)
    assert np.array_equal(oracle.bf16_round(f32(y32)).view(np.uint32), f32(y).view(np.uint32))
    host_sum = oracle.bf16_round(np.float32(f32(y32)) + np.float32(f32(r)))
    assert np.array_equal(host_sum.view(np.uint32), f32(yr).view(np.uint32))


def test_random_dense_cover_both_tails():
    """The drawn shapes include K tails that are split and ones that are not
    (the workspace query says which, without launching anything)."""
    split = [fb.fp8_blockscaled_gemm_workspace_bytes(*_draw_dense(kind, seed)[:3]) > 0 for kind, seed in _DENSE]
    assert any(split) and not all(split), split


def _draw_counts(rng):
    G = int(rng.integers(1, 11))
    counts = []
    for _ in range(G):
        u = rng.uniform()
        if u < 0.15:
            counts.append(0)
        elif u < 0.5:
            counts.append(int(rng.integers(1, 131)))
        elif u < 0.8:
            counts.append(max(0, 256 * int(rng.integers(1, 4)) + int(rng.integers(-2, 3))))
        else:
            counts.append(int(rng.integers(1, 701)))
    return counts


@pytest.mark.parametrize("seed", [2000, 2001, 2002, 2003, 2004, 2005])
def test_random_grouped(seed):
    rng = np.random.default_rng(seed)
    counts = _draw_counts(rng)
    G = len(counts)
    N = 128 * int(rng.choice([1, 2, 3, 4, 8]))
    K = 128 * int(rng.integers(1, 7))
    offsets = workloads.grouped_offsets(counts)
    m_total = int(offsets[-1])
    x, _ = workloads.dense_inputs(max(m_total, 1), 128, K, seed=seed)
    x = x[:m_total]
    _, w = workloads.dense_inputs(1, G * N, K, seed=seed + 1)
    w = w.reshape(G, N, K)
    qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    y = fb.fp8_blockscaled_grouped_gemm(offsets.to(DEV), m_total, qa, sa, qw, sw)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    what = f"counts={counts} N={N} K={K}"
    qa_r, sa_r = oracle.quant_act_1x128(f32(x))
    qw_r, sw_r = oracle.quant_weight_128x128(f32(w).reshape(G * N, K))
    assert_codes_equal(u8(qa), qa_r, f"qa {what}")
    assert_scales_equal(f32(sa)[:, :m_total], sa_r, f"sa {what}")
    assert_codes_equal(u8(qw).reshape(G * N, K), qw_r, f"qw {what}")
    assert_scales_equal(f32(sw).reshape(G * N // 128, K // 128), sw_r, f"sw {what}")
    y_ref = oracle.blockscaled_grouped_gemm(offsets.numpy(), qa_r, sa_r, qw_r.reshape(G, N, K),
                                            sw_r.reshape(G, N // 128, K // 128))
    assert_gemm_close(f32(y), y_ref, what=f"grouped {what}")


@pytest.mark.parametrize("seed", [3000, 3001, 3002, 3003, 3004, 3005])
def test_random_quant(seed):
    """Both quantisers on drawn shapes, with row magnitudes spread over 2^-60
    .. 2^60 (every row's scale far from the others')."""
    rng = np.random.default_rng(seed)
    M = int(rng.integers(1, 3001))
    K = 128 * int(rng.integers(1, 33))
    N = 128 * int(rng.integers(1, 33))
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= (2.0 ** rng.integers(-60, 61, size=(M, 1))).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 10.0 ** rng.uniform(-3, 1)).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    wb = torch.from_numpy(w).to(torch.bfloat16)
    qa, sa = fb.fp8_quant_act_1x128(xb.to(DEV))
    qw, sw = fb.fp8_quant_weight_128x128(wb.to(DEV))
    torch.cuda.synchronize()
    qa_r, sa_r = oracle.quant_act_1x128(f32(xb))
    qw_r, sw_r = oracle.quant_weight_128x128(f32(wb))
    assert_codes_equal(u8(qa), qa_r, f"qa M={M} K={K}")
    assert_scales_equal(f32(sa)[:, :M], sa_r, f"sa M={M} K={K}")
    assert_codes_equal(u8(qw), qw_r, f"qw N={N} K={K}")
    assert_scales_equal(f32(sw), sw_r, f"sw N={N} K={K}")


@pytest.mark.parametrize("seed", [4000, 4001, 4002, 4003, 4004])
def test_random_backward(seed):
    """Both backward GEMMs on drawn shapes (tokens M a multiple of 128, the
    weight-gradient contraction), with X in BF16 and from its FP8 forward
    cache ("The Definitive Information To Deepseek", paragraphs 2 and 3)."""
    rng = np.random.default_rng(seed)
    while True:
        M = 128 * int(rng.integers(1, 17))
        N = 128 * int(rng.integers(1, 25))
        K = 128 * int(rng.integers(1, 17))
        if M * N * K <= 3e9:
            break
    x, w, dy = workloads.backward_inputs(M, N, K, seed=seed, w_std=float(10.0 ** rng.uniform(-3, 0)))
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    dx, dw = fb.linear_backward(xd, wd, dyd)
    qa, sa = fb.fp8_quant_act_1x128(xd)
    dx_c, dw_c = fb.linear_backward(None, wd, dyd, x_cache=(qa, sa))
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    what = f"M={M} N={N} K={K}"
    dx_ref, dw_ref = oracle.linear_backward(f32(x), f32(w), f32(dy))
    assert_gemm_close(f32(dx), dx_ref, what=f"dX {what}")
    assert_gemm_close(f32(dw), dw_ref, what=f"dW {what}")
    qa_r, sa_r = oracle.quant_act_1x128(f32(x))
    _, dw_c_ref = oracle.linear_backward_cached(qa_r, sa_r, f32(w), f32(dy))
    assert torch.equal(dx_c, dx)  # dX does not depend on where X comes from
    assert_gemm_close(f32(dw_c), dw_c_ref, what=f"dW from the FP8 cache {what}")


@pytest.mark.parametrize("seed", [5000, 5001, 5002, 5003])
def test_random_packed(seed):
    """The GEMM on packed weight tiles, on drawn skinny shapes (the
    weight-streaming case it serves): within the GEMM tolerance of the
    oracle."""
    rng = np.random.default_rng(seed)
    M = int(rng.integers(1, 129))
    N = 128 * int(rng.integers(1, 49))
    K = 128 * int(rng.integers(1, 33))
    x, w = workloads.dense_inputs(M, N, K, seed=seed)
    qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    wp = fb.fp8_pack_weight_128x128(qw)
    y = fb.fp8_blockscaled_gemm_packed(qa, sa, wp, sw)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    y_ref, _ = oracle.linear_forward(f32(x), f32(w))
    assert_gemm_close(f32(y), y_ref, what=f"packed M={M} N={N} K={K}")


@pytest.mark.parametrize("seed", [6000, 6001, 6002, 6003, 6004])
def test_random_per_token_and_per_channel(seed):
    """The per-token and per-channel quantisers on drawn shapes (K a multiple
    of 8), rows and columns of widely spread magnitudes, bit for bit."""
    rng = np.random.default_rng(seed)
    M = int(rng.integers(1, 5001))
    K = 8 * int(rng.integers(1, 513))
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= (2.0 ** rng.integers(-40, 41, size=(M, 1))).astype(np.float32)
    x *= (2.0 ** rng.integers(-20, 21, size=(1, K))).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    xd = xb.to(DEV)
    qt, st = fb.fp8_quant_per_token(xd)
    qc, sc = fb.fp8_quant_per_channel(xd)
    torch.cuda.synchronize()
    qt_r, st_r = oracle.quant_per_token(f32(xb))
    qc_r, sc_r = oracle.quant_per_channel(f32(xb))
    assert_codes_equal(u8(qt), qt_r, f"per-token codes M={M} K={K}")
    assert_scales_equal(f32(st), st_r, f"per-token scales M={M} K={K}")
    assert_codes_equal(u8(qc), qc_r, f"per-channel codes M={M} K={K}")
    assert_scales_equal(f32(sc), sc_r, f"per-channel scales M={M} K={K}")


@pytest.mark.parametrize("seed", [7000, 7001, 7002, 7003])
def test_random_transposed_operands(seed):
    """The weight-gradient operands on drawn shapes: 1x128 tiles of X^T from
    BF16 X and from X's FP8 cache (dequantised to BF16, then requantised),
    the 128x128 code and scale transpose of W, and the block dequant of W,
    all bit for bit."""
    rng = np.random.default_rng(seed)
    M = 128 * int(rng.integers(1, 25))
    K = 128 * int(rng.integers(1, 41))
    N = 128 * int(rng.integers(1, 25))
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= (2.0 ** rng.integers(-30, 31, size=(1, K))).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    _, w = workloads.dense_inputs(1, N, K, seed=seed, w_std=float(10.0 ** rng.uniform(-3, 1)))
    xd = xb.to(DEV)
    qxt, sxt = fb.fp8_quant_act_1x128_t(xd)
    qa, sa = fb.fp8_quant_act_1x128(xd)
    qrt, srt = fb.fp8_requant_act_1x128_t(qa, sa)
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    qwt, swt = fb.fp8_transpose_weight_128x128(qw, sw)
    wd = fb.fp8_dequant_weight_128x128(qw, sw)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    what = f"M={M} N={N} K={K}"
    q_ref, s_ref = oracle.quant_act_1x128_t(f32(xb))
    assert_codes_equal(u8(qxt), q_ref, f"codes of x^T {what}")
    assert_scales_equal(f32(sxt)[:, :K], s_ref, f"scales of x^T {what}")
    qa_r, sa_r = oracle.quant_act_1x128(f32(xb))
    qr_ref, sr_ref = oracle.requant_act_1x128_t(qa_r, sa_r)
    assert_codes_equal(u8(qrt), qr_ref, f"requantised codes {what}")
    assert_scales_equal(f32(srt)[:, :K], sr_ref, f"requantised scales {what}")
    qw_r, sw_r = oracle.quant_weight_128x128(f32(w))
    qwt_r, swt_r = oracle.transpose_weight_128x128(qw_r, sw_r)
    assert_codes_equal(u8(qwt), qwt_r, f"codes of W^T {what}")
    assert_scales_equal(f32(swt), swt_r, f"scales of W^T {what}")
    wd_ref = oracle.dequant_weight_128x128_bf16(qw_r, sw_r)
    assert np.array_equal(f32(wd).view(np.uint32), wd_ref.view(np.uint32)), f"dequant {what}"


@pytest.mark.parametrize("seed", [8000, 8001, 8002])
def test_random_e5m6_and_swiglu(seed):
    """E5M6 round trips of drawn lengths (a multiple of 8), and the SwiGLU +
    1x128 quantiser on drawn shapes: codes bit for bit given the kernel's own
    BF16 product, which stays within a few ulps of the float64 product."""
    rng = np.random.default_rng(seed)
    n = 8 * int(rng.integers(1, 200001))
    v = (rng.standard_normal(n) * 2.0 ** rng.integers(-20, 21, size=n)).astype(np.float32)
    vb = torch.from_numpy(v).to(torch.bfloat16)
    codes = fb.e5m6_encode(vb.to(DEV))
    back = fb.e5m6_decode(codes)
    M = int(rng.integers(1, 3001))
    F = 128 * int(rng.integers(1, 25))
    gu = torch.from_numpy((rng.standard_normal((M, 2 * F)) * 3.0).astype(np.float32)).to(torch.bfloat16)
    qa, sa, h = fb.fp8_swiglu_quant_act_1x128(gu.to(DEV), return_h=True)
    torch.cuda.synchronize()
    vf = f32(vb)
    want = oracle.e5m6_encode_rne_satfinite(vf)
    assert np.array_equal(codes.cpu().numpy().view(np.uint16), want), f"e5m6 codes n={n}"
    assert np.array_equal(f32(back).astype(np.float64), oracle.e5m6_decode(want)), f"e5m6 decode n={n}"
    hg = f32(h)
    q_ref, s_ref = oracle.quant_act_1x128(hg)
    assert_codes_equal(u8(qa), q_ref, f"swiglu codes M={M} F={F}")
    assert_scales_equal(f32(sa)[:, :M], s_ref, f"swiglu scales M={M} F={F}")
    guf = f32(gu)
    h64 = oracle.silu_mul(guf[:, :F], guf[:, F:])
    a = np.abs(h64)
    ulp_bf16 = 2.0 ** (np.floor(np.log2(np.maximum(a, 1e-38))) - 7)
    assert np.all(np.abs(hg - h64) <= 0.5 * ulp_bf16 + a * 2.0 ** -20), f"swiglu product M={M} F={F}"
