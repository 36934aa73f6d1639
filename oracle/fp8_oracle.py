"""Plain CPU oracle for the fine-grained FP8 block-scaled linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests, the smoke check and the benchmark's CPU
baseline leg use it.  It shares no code, table or constant generator with the
CUDA library; it is a slow, direct restatement of the method so that a reader
can check it against the source text by eye.

Source: the DeepSeek-V3 FP8 mixed-precision framework excerpt reposted as
"The Definitive Information To Deepseek":
  * paragraph 3, "Figure 7 (a)" items (1) and (2): activations are grouped and
    scaled on 1x128 tiles (per token per 128 channels), weights on 128x128
    blocks (per 128 input channels per 128 output channels);
  * paragraph 2, last sentence: a scaling factor is derived per group and the
    activation or weight is quantised online into FP8;
  * paragraph 4, first sentence: the GEMMs take FP8 tensors and produce BF16
    (or FP32) outputs;
  * paragraph 1, last sentence: partial sums are promoted (moved to a higher
    precision accumulator) while the next MMA runs.

Where the excerpt is silent the plainest reading is taken:
  * the FP8 format is OCP E4M3FN (bias 7, largest finite 448, no infinities);
  * the per-group statistic is the maximum absolute value (amax) and the FP32
    scale is s = fl32(amax / 448); values are quantised as E4M3(fl32(x / s))
    with round-to-nearest-even and saturation to +-448 (never NaN);
  * an all-zero group has s = 0 and every code +0 (0x00);
  * a value of a non-zero group that rounds to zero keeps its sign (0x80);
  * promotion happens once per 128-wide K chunk, i.e. exactly at the scale
    group boundaries, so
        Y[m, n] = sum_kb  sa[kb, m] * sw[n // 128, kb]
                          * sum_{k in chunk kb} dec(qa[m, k]) * dec(qw[n, k]);
  * scales are laid out sa[kb, m] (token index contiguous) and
    sw[nb, kb] (row-major over weight blocks).

Precision: E4M3 products have at most 8 significant bits and lie in
[2**-18, 448**2]; a sum of 128 of them fits in 43 bits, so every chunk sum
below is exact in float64 whatever order the BLAS routine adds in.  The
scales are float32, so sa * sw is exact in float64 too; only the final sum
over K chunks rounds (at float64 precision).

Rounded float32 division fl32(a / b) is computed as float32(float64(a) /
float64(b)).  Rounding a quotient first to 53 and then to 24 bits gives the
correctly rounded 24-bit quotient because 53 >= 2 * 24 + 2 (S. A. Figueroa,
"When is double rounding innocuous?", SIGNUM Newsletter 30(3), 1995); the
tests pin this against exact rational arithmetic.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0  # largest finite E4M3FN magnitude, code S.1111.110
GROUP = 128       # group width along K (and block height along N for weights)


# ---------------------------------------------------------------------------
# E4M3FN codec, written from the format definition.
# ---------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Exact float64 value of each OCP E4M3FN byte.

    Layout S.EEEE.MMM with exponent bias 7:
      E > 0 : (-1)**S * 2**(E - 7) * (1 + M / 8)
      E = 0 : (-1)**S * 2**(-6)    * (M / 8)       (subnormals and +-0)
      E = 15, M = 7 : NaN (the only non-finite codes, 0x7F and 0xFF).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = c >> 7
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = np.ldexp(1.0 + man / 8.0, exp - 7)
    subnormal = np.ldexp(man / 8.0, -6)
    mag = np.where(exp == 0, subnormal, normal)
    mag = np.where((exp == 15) & (man == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


# Non-negative finite codes 0x00 .. 0x7E.  Their values increase with the
# code, so consecutive codes are neighbouring representable values.
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = e4m3_decode(_POS_CODES.astype(np.uint8))


def e4m3_encode_rne_satfinite(v) -> np.ndarray:
    """E4M3FN code of each float32 value: nearest representable value, ties to
    the even code (mantissa LSB 0), magnitudes above 448 saturate to 448.

    The sign is the sign bit of the input, so -0.0 and negative values that
    round to zero both give 0x80.  NaN inputs are outside the contract.
    """
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v).astype(np.float64)
    # hi is the first non-negative code whose value is >= a.
    hi = np.searchsorted(_POS_VALUES, a, side="left")
    saturate = hi >= len(_POS_VALUES)  # a > 448
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS_VALUES[hi] - a  # exact: both operands are short dyadic numbers
    d_lo = a - _POS_VALUES[lo]
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(saturate, 0x7E, code)
    code = code | (np.signbit(v).astype(np.int64) << 7)
    return code.astype(np.uint8)


# ---------------------------------------------------------------------------
# Rounded float32 arithmetic.
# ---------------------------------------------------------------------------

def fl32_div(a, b) -> np.ndarray:
    """Correctly rounded float32 quotient a / b of float32 operands (see the
    module docstring for why the float64 detour is exact).  b == 0 gives a
    non-finite result that callers never use."""
    a64 = np.asarray(a, dtype=np.float32).astype(np.float64)
    b64 = np.asarray(b, dtype=np.float32).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        return (a64 / b64).astype(np.float32)


# ---------------------------------------------------------------------------
# Group quantisation ("Figure 7 (a)" grouping + online scaling).
# ---------------------------------------------------------------------------

def _quantise_groups(g: np.ndarray):
    """Quantise every group along the last axis of ``g`` (float32).

    Returns (codes uint8 with the shape of g, scales float32 with g.shape[:-1]).
    """
    amax = np.max(np.abs(g), axis=-1)            # exact in float32
    s = fl32_div(amax, np.float32(E4M3_MAX))     # s = fl32(amax / 448)
    v = fl32_div(g, s[..., None])                # fl32(x / s)
    codes = e4m3_encode_rne_satfinite(v)
    codes[s == 0] = 0                            # all-zero group: every code +0
    return codes, s


def quant_act_1x128(x):
    """1x128 activation quantisation (one scale per token per 128 channels).

    x  : float32 [M, K] holding BF16 values, K % 128 == 0.
    Returns qa uint8 [M, K] (E4M3FN codes) and sa float32 [K/128, M]
    (sa[kb, m] is the scale of row m, channels 128*kb .. 128*kb + 127).
    """
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    codes, s = _quantise_groups(x.reshape(M, K // GROUP, GROUP))
    return codes.reshape(M, K), np.ascontiguousarray(s.T)


def quant_weight_128x128(w):
    """128x128 weight quantisation (one scale per 128 output x 128 input
    channels).

    w  : float32 [N, K] holding BF16 values (row n = output channel n),
         N % 128 == 0, K % 128 == 0.
    Returns qw uint8 [N, K] and sw float32 [N/128, K/128]
    (sw[nb, kb] covers rows 128*nb.. and columns 128*kb..).
    """
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    if N % GROUP or K % GROUP:
        raise ValueError("N and K must be multiples of 128")
    NB, KB = N // GROUP, K // GROUP
    # [NB, 128, KB, 128] -> [NB, KB, 128*128]: one row per block.
    blocks = w.reshape(NB, GROUP, KB, GROUP).transpose(0, 2, 1, 3).reshape(NB, KB, GROUP * GROUP)
    codes, s = _quantise_groups(blocks)
    qw = codes.reshape(NB, KB, GROUP, GROUP).transpose(0, 2, 1, 3).reshape(N, K)
    return np.ascontiguousarray(qw), s


def dequant_weight_128x128(qw, sw):
    """float64 W ~= dec(qw) * sw broadcast over each 128x128 block."""
    qw = np.asarray(qw, dtype=np.uint8)
    N, K = qw.shape
    scale = np.repeat(np.repeat(np.asarray(sw, dtype=np.float64), GROUP, axis=0), GROUP, axis=1)
    return e4m3_decode(qw) * scale


def bf16_round(v) -> np.ndarray:
    """float32 -> nearest BF16 value (ties to the even BF16 significand),
    returned as float32.  BF16 keeps the top 16 bits of a float32; rounding
    adds half a BF16 ulp minus one, plus the parity of the kept LSB, before
    truncating.  Finite inputs only."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (r.astype(np.uint32) << 16).view(np.float32)


def dequant_weight_128x128_bf16(qw, sw):
    """BF16 weights back from 128x128-quantised codes: for each element,
    bf16(fl32(dec(q) * s)) with s its block's scale -- the float32 product of
    the exact code value and the scale, rounded to BF16: the FP8-to-BF16
    weight conversion that the DeepSeek-V3 model card (section 6, "How to Run
    Locally") offers for its FP8-only release.  Reading: the product is
    formed in float32 and rounded to nearest even BF16.
    Returns float32 [N, K] holding BF16 values."""
    qw = np.asarray(qw, dtype=np.uint8)
    scale = np.repeat(np.repeat(np.asarray(sw, dtype=np.float32), GROUP, axis=0), GROUP, axis=1)
    prod = e4m3_decode(qw).astype(np.float32) * scale  # float32 multiply, rounded once
    return bf16_round(prod)


# ---------------------------------------------------------------------------
# Block-scaled GEMM with per-128-K-chunk promotion.
# ---------------------------------------------------------------------------

def blockscaled_gemm(qa, sa, qw, sw):
    """Y[m, n] = sum_kb sa[kb, m] * sw[n//128, kb] * (chunk kb of dec(qa) . dec(qw)^T).

    qa uint8 [M, K], sa float32 [K/128, M], qw uint8 [N, K], sw float32
    [N/128, K/128].  Returns float64 [M, N], unrounded (the GPU writes BF16).
    """
    qa = np.asarray(qa, dtype=np.uint8)
    qw = np.asarray(qw, dtype=np.uint8)
    sa = np.asarray(sa, dtype=np.float32)
    sw = np.asarray(sw, dtype=np.float32)
    M, K = qa.shape
    N = qw.shape[0]
    KB = K // GROUP
    y = np.zeros((M, N), dtype=np.float64)
    for kb in range(KB):
        cols = slice(kb * GROUP, (kb + 1) * GROUP)
        a = e4m3_decode(qa[:, cols])
        b = e4m3_decode(qw[:, cols])
        chunk = a @ b.T                                           # exact
        row_scale = sa[kb, :M].astype(np.float64)                 # [M]
        col_scale = np.repeat(sw[:, kb].astype(np.float64), GROUP)  # [N]
        y += chunk * (row_scale[:, None] * col_scale[None, :])    # promotion
    return y


def blockscaled_gemm_residual(qa, sa, qw, sw, r):
    """The block-scaled GEMM with a residual added before the output rounding:
    Y = (sum of the promoted chunks) + R, R a BF16 [M, N] matrix given as
    float values, in float64.  Reading: the residual stream of the block is
    added to the linear layer's FP32 result in the epilogue, and the sum is
    rounded once to the output format ("outputs in BF16 or FP32",
    paragraph 4 of "The Definitive Information To Deepseek").  Returns float64
    [M, N], unrounded."""
    return blockscaled_gemm(qa, sa, qw, sw) + np.asarray(r, dtype=np.float64)


def blockscaled_grouped_gemm(offsets, qa, sa, qw, sw):
    """Grouped (per-expert) block-scaled GEMM.

    Rows offsets[g] .. offsets[g+1]-1 of qa / sa / Y belong to group g and are
    multiplied by weight group g.  qw uint8 [G, N, K], sw float32
    [G, N/128, K/128], offsets int [G+1] with offsets[0] == 0, non-decreasing.
    Returns float64 [offsets[G], N].
    """
    offsets = [int(o) for o in offsets]
    qa = np.asarray(qa, dtype=np.uint8)
    sa = np.asarray(sa, dtype=np.float32)
    G = len(offsets) - 1
    N = qw.shape[1]
    y = np.zeros((offsets[-1], N), dtype=np.float64)
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 > r0:
            y[r0:r1] = blockscaled_gemm(qa[r0:r1], sa[:, r0:r1], qw[g], sw[g])
    return y


# ---------------------------------------------------------------------------
# Quantisation variants.  The TileKernels release ("DeepSeek starts updating
# frequently", section on the tile kernels' features, item "Quantification")
# converts to FP8/FP4/E5M6 "per token", "per block" and "per channel" and fuses
# SwiGLU with the quantisation; the V3 excerpt keeps certain activations in a
# custom E5M6 format (paragraph 3).  Readings: per token = one scale per row
# of X [tokens, channels] over all its channels; per channel = one scale per
# column over all tokens; both with the same amax / 448 rule as the 1x128
# tiles.
# ---------------------------------------------------------------------------

def quant_per_token(x):
    """One FP32 scale per row: codes [M, K], scales [M]."""
    x = np.asarray(x, dtype=np.float32)
    return _quantise_groups(x)


def quant_per_channel(x):
    """One FP32 scale per column: codes [M, K], scales [K]."""
    x = np.asarray(x, dtype=np.float32)
    codes, s = _quantise_groups(np.ascontiguousarray(x.T))
    return np.ascontiguousarray(codes.T), s


def silu_mul(gate, up):
    """SwiGLU's product silu(g) * u = g / (1 + exp(-g)) * u in float64."""
    g = np.asarray(gate, dtype=np.float64)
    u = np.asarray(up, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def swiglu_quant_act_1x128(gate_up):
    """SwiGLU then 1x128 quantisation.  gate_up float32 [M, 2F] holds the
    gate in columns [0, F) and the up projection in [F, 2F) (BF16 values).
    Reading: h = silu(g) * u is rounded to BF16 -- the activation the
    quantiser sees is the one an unfused pipeline would store -- and then
    quantised exactly as quant_act_1x128.  Returns (h float32 [M, F] holding
    BF16 values, codes [M, F], scales [F/128, M])."""
    gu = np.asarray(gate_up, dtype=np.float32)
    F = gu.shape[1] // 2
    h = bf16_round(silu_mul(gu[:, :F], gu[:, F:]).astype(np.float32))
    qa, sa = quant_act_1x128(h)
    return h, qa, sa


# E5M6: sign, 5 exponent bits (bias 15), 6 mantissa bits in the low 12 bits of
# a 16-bit word.  Reading (the pages give the name only): IEEE-style like
# FP16 with the mantissa cut to 6 bits -- subnormals 2^-14 * m / 64, exponent
# field 31 reserved (decoded as inf / NaN) -- encoded with round-to-nearest-
# even and saturation to the largest finite value (1 + 63/64) * 2^15 = 65024,
# without a scale factor.
E5M6_MAX = 65024.0


def e5m6_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint16).astype(np.int64) & 0xFFF
    sign = c >> 11
    exp = (c >> 6) & 0x1F
    man = c & 0x3F
    normal = np.ldexp(1.0 + man / 64.0, exp - 15)
    subnormal = np.ldexp(man / 64.0, -14)
    mag = np.where(exp == 0, subnormal, normal)
    mag = np.where(exp == 31, np.where(man == 0, np.inf, np.nan), mag)
    return np.where(sign == 1, -mag, mag)


_E5M6_POS_CODES = np.arange(31 << 6, dtype=np.int64)  # 0x000 .. 0x7BF, all finite non-negative
_E5M6_POS_VALUES = e5m6_decode(_E5M6_POS_CODES.astype(np.uint16))


def e5m6_encode_rne_satfinite(v) -> np.ndarray:
    """E5M6 code of each float32 value: nearest representable value, ties to
    the even code, magnitudes above 65024 saturate; the sign bit follows the
    input's.  NaN inputs are outside the contract."""
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v).astype(np.float64)
    hi = np.searchsorted(_E5M6_POS_VALUES, a, side="left")
    saturate = hi >= len(_E5M6_POS_VALUES)
    hi = np.minimum(hi, len(_E5M6_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E5M6_POS_VALUES[hi] - a
    d_lo = a - _E5M6_POS_VALUES[lo]
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_E5M6_POS_CODES[hi] % 2 == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(saturate, len(_E5M6_POS_VALUES) - 1, code)
    code = code | (np.signbit(v).astype(np.int64) << 11)
    return code.astype(np.uint16)


# ---------------------------------------------------------------------------
# Backward GEMMs of the FP8 linear layer.
#
# The excerpt trains with the same FP8 GEMMs: the activation is cached in FP8
# for the backward pass of the linear layer (paragraph 2) and the backward is
# split into the input-gradient and weight-gradient parts (paragraph 3).
#   dX = dY . W        : dY quantised 1x128 along N (its reduction dim), W's
#                        128x128 blocks transposed (a block is a block either
#                        way round, so the codes and scales just move);
#   dW = dY^T . X      : the reduction runs over tokens, so both operands are
#                        quantised 1x128 along M -- the 1x128 quantisation of
#                        the transposed matrices -- and each chunk is promoted
#                        with one scale per output row times one per column.
# ---------------------------------------------------------------------------

def quant_act_1x128_t(x):
    """1x128 quantisation of x^T: for each column k of x [M, K] and each run
    of 128 rows, one scale.  Returns codes [K, M] (x^T's layout) and scales
    [M/128, K] (the activation-scale layout of x^T).  M % 128 == 0."""
    x = np.asarray(x, dtype=np.float32)
    return quant_act_1x128(np.ascontiguousarray(x.T))


def transpose_weight_128x128(qw, sw):
    """Codes and block scales of W^T from those of W: qw^T [K, N], sw^T
    [K/128, N/128]."""
    return np.ascontiguousarray(np.asarray(qw, dtype=np.uint8).T), np.ascontiguousarray(np.asarray(sw).T)


def blockscaled_gemm_rowscaled(qa, sa, qb, sb):
    """Y[m, n] = sum_kb sa[kb, m] * sb[kb, n] * (chunk kb of dec(qa) . dec(qb)^T)
    with 1x128 scales on both operands (the weight-gradient GEMM).
    qa uint8 [M, K], sa float32 [K/128, >=M], qb uint8 [N, K], sb float32
    [K/128, >=N].  Returns float64 [M, N], unrounded."""
    qa = np.asarray(qa, dtype=np.uint8)
    qb = np.asarray(qb, dtype=np.uint8)
    sa = np.asarray(sa, dtype=np.float32)
    sb = np.asarray(sb, dtype=np.float32)
    M, K = qa.shape
    N = qb.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    for kb in range(K // GROUP):
        cols = slice(kb * GROUP, (kb + 1) * GROUP)
        chunk = e4m3_decode(qa[:, cols]) @ e4m3_decode(qb[:, cols]).T          # exact
        y += chunk * (sa[kb, :M].astype(np.float64)[:, None] * sb[kb, :N].astype(np.float64)[None, :])
    return y


def linear_backward(x, w, dy):
    """Both backward GEMMs on float32 inputs holding BF16 values:
    dX = Q(dY) . Q(W)^T-blocks and dW = Q(dY^T) . Q(X^T)^T.
    Returns (dx float64 [M, K], dw float64 [N, K])."""
    return _linear_backward_from(quant_act_1x128_t(x), w, dy)


def _linear_backward_from(xt, w, dy):
    """The two backward GEMMs given X's weight-gradient operand xt = (codes
    [K, M], scales [M/128, K])."""
    qw, sw = quant_weight_128x128(w)
    qdy, sdy = quant_act_1x128(dy)
    qwt, swt = transpose_weight_128x128(qw, sw)
    dx = blockscaled_gemm(qdy, sdy, qwt, swt)
    qdyt, sdyt = quant_act_1x128_t(dy)
    qxt, sxt = xt
    dw = blockscaled_gemm_rowscaled(qdyt, sdyt, qxt, sxt)
    return dx, dw


def dequant_act_1x128_bf16(qa, sa):
    """BF16 activation back from its cached 1x128 FP8 form: for each element,
    bf16(fl32(dec(qa[m, k]) * sa[k // 128, m])), the same float32 product
    and single BF16 rounding as dequant_weight_128x128_bf16 with the 1x128
    grouping.  qa uint8 [M, K], sa float32 [K/128, >=M].  Returns float32
    [M, K] holding BF16 values."""
    qa = np.asarray(qa, dtype=np.uint8)
    M, K = qa.shape
    sa = np.asarray(sa, dtype=np.float32)[:, :M]
    scale = np.repeat(np.ascontiguousarray(sa.T), GROUP, axis=1)   # [M, K]: row m, chunk k // 128
    prod = e4m3_decode(qa).astype(np.float32) * scale              # float32 multiply, rounded once
    x = bf16_round(prod)
    return x


def requant_act_1x128_t(qa, sa):
    """The weight-gradient operand from the activation cached in FP8 for the
    backward pass (paragraph 2 of "The Definitive Information To Deepseek"):
    the cached 1x128 codes are dequantised to BF16 (above), and that matrix
    is quantised on 1x128 tiles of its transpose (per channel per 128
    tokens), exactly as quant_act_1x128_t does for a BF16 activation.
    Returns codes [K, M] and scales [M/128, K].  M % 128 == 0."""
    return quant_act_1x128_t(dequant_act_1x128_bf16(qa, sa))


def linear_backward_cached(qa, sa, w, dy):
    """linear_backward with the activation taken from its cached FP8 form
    (qa, sa) -- the forward's 1x128 quantisation of X -- instead of BF16 X:
    dW = Q(dY^T) . R(qa, sa)^T with R = requant_act_1x128_t; dX as in
    linear_backward.  Returns (dx float64 [M, K], dw float64 [N, K])."""
    return _linear_backward_from(requant_act_1x128_t(qa, sa), w, dy)


def linear_forward(x, w):
    """The whole hot path on float32 inputs holding BF16 values: quantise X
    per 1x128 tile and W per 128x128 block, then the block-scaled GEMM."""
    qa, sa = quant_act_1x128(x)
    qw, sw = quant_weight_128x128(w)
    return blockscaled_gemm(qa, sa, qw, sw), (qa, sa, qw, sw)
