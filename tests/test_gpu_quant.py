"""Bit-exact parity of the CUDA quantisation kernels with the CPU oracle.

1x128 activation tiles and 128x128 weight blocks ("The Definitive
Information To Deepseek", paragraph 3, "Figure 7 (a)"); per-group online
scale (paragraph 2).  Codes and scales must match bit for bit.
"""
import numpy as np
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
import oracle
from fp8_fine_grained_14_b300 import workloads
from helpers import assert_codes_equal, assert_scales_equal, f32, u8
from oracle_pins import exact_tie_groups

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _act_parity(x_cpu, rows=None):
    x = x_cpu.to(DEV)
    qa, sa = fb.fp8_quant_act_1x128(x)
    torch.cuda.synchronize()
    M = x_cpu.shape[0]
    rows = np.arange(M) if rows is None else rows
    qa_ref, sa_ref = oracle.quant_act_1x128(f32(x_cpu)[rows])
    assert_codes_equal(u8(qa)[rows], qa_ref, "qa")
    assert_scales_equal(f32(sa)[:, rows], sa_ref, "sa")
    return qa, sa


def _weight_parity(w_cpu, blocks=None):
    w = w_cpu.to(DEV)
    qw, sw = fb.fp8_quant_weight_128x128(w)
    torch.cuda.synchronize()
    if w_cpu.dim() == 3:
        G, N, K = w_cpu.shape
        w2, qw2, sw2 = w_cpu.reshape(G * N, K), qw.reshape(G * N, K), sw.reshape(G * N // 128, K // 128)
    else:
        w2, qw2, sw2 = w_cpu, qw, sw
    NB = w2.shape[0] // 128
    blocks = np.arange(NB) if blocks is None else blocks
    rows = np.concatenate([np.arange(b * 128, b * 128 + 128) for b in blocks])
    qw_ref, sw_ref = oracle.quant_weight_128x128(f32(w2)[rows])
    assert_codes_equal(u8(qw2)[rows], qw_ref, "qw")
    assert_scales_equal(f32(sw2)[blocks], sw_ref, "sw")
    return qw, sw


@pytest.mark.parametrize("M,K", [(128, 256), (1, 128), (3, 384), (127, 128), (129, 640), (300, 896), (1000, 1280)])
def test_act_quant_shapes(M, K):
    x, _ = workloads.dense_inputs(M, 128, K, seed=M + K)
    _act_parity(x)


@pytest.mark.parametrize("N,K", [(128, 128), (256, 256), (384, 640), (1024, 1152)])
def test_weight_quant_shapes(N, K):
    _, w = workloads.dense_inputs(1, N, K, seed=N + K)
    _weight_parity(w)


def test_act_quant_exact_ties_and_edges():
    """Exact E4M3 midpoint quotients, all-zero groups (with -0), tiny
    (subnormal-scale) and huge groups, negative values rounding to zero."""
    # exact-tie rows: BF16 holds m*s exactly for these short-mantissa scales
    x_ties, _ = exact_tie_groups(scales=(1.5, 1.75, 1.25, 0.75 * 2.0 ** -20, 1.5 * 2.0 ** 30))
    ties_bf16 = torch.from_numpy(x_ties).to(torch.bfloat16)
    assert np.array_equal(f32(ties_bf16), x_ties), "tie inputs must be BF16-exact"
    rows = [x_ties]
    rng = np.random.default_rng(0)
    z = np.zeros((1, 128), dtype=np.float32)
    z[0, 5] = -0.0
    rows.append(z)
    # -126 .. -60: scales far below 2^-64 (IEEE division path); -58 .. -52:
    # amax around 448 * 2^-64, where the exact FMA-corrected quotient takes over
    for e in (-133, -126, -120, -60, -58, -57, -56, -55, -54, -52, 60, 120):
        rows.append((rng.standard_normal((1, 128)) * 2.0 ** e).astype(np.float32))
    negz = rng.standard_normal((1, 128)).astype(np.float32)
    negz[0, 3:9] = -0.0  # -0 inside a non-zero group codes as 0x80
    rows.append(negz)
    mixed = rng.standard_normal((1, 128)).astype(np.float32)
    mixed[0, :10] = -(2.0 ** -20)  # far below the group's E4M3 resolution: -0 codes
    rows.append(mixed)
    x = torch.from_numpy(np.concatenate(rows)).to(torch.bfloat16)
    qa, _ = _act_parity(x)
    assert u8(qa)[len(x_ties), 5] == 0x00  # -0 in an all-zero group codes as +0
    assert np.all(u8(qa)[-2, 3:9] == 0x80)
    assert np.all(u8(qa)[-1, :10] == 0x80)


def test_weight_quant_edges():
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((512, 256)) * 0.02).astype(np.float32)
    w[0:128, 0:128] = 0.0                # all-zero block
    w[128:256, 128:256] *= 2.0 ** -126   # tiny block (subnormal scale)
    w[256:384, 0:128] *= 2.0 ** 100      # huge block
    w[384:512, 128:256] = 448.0 * 1.5    # constant block, s = 1.5
    _weight_parity(torch.from_numpy(w).to(torch.bfloat16))


def test_act_quant_strided_input_and_ld_sa():
    """Row strides larger than K and a padded scale stride."""
    x_full, _ = workloads.dense_inputs(200, 128, 512, seed=3)
    xd = x_full.to(DEV)[:, :384]  # ldx = 512, K = 384
    qa = torch.full((200, 400), 0x55, dtype=torch.uint8, device=DEV)[:, :384]  # ldq = 400
    sa = torch.full((3, 208), -1.0, dtype=torch.float32, device=DEV)
    fb.fp8_quant_act_1x128(xd, qa=qa, sa=sa)
    torch.cuda.synchronize()
    qa_ref, sa_ref = oracle.quant_act_1x128(f32(x_full)[:, :384])
    assert_codes_equal(u8(qa), qa_ref, "qa")
    assert_scales_equal(f32(sa)[:, :200], sa_ref, "sa")
    assert np.all(f32(sa)[:, 200:] == -1.0), "columns >= M of sa must be untouched"


def inexact_scale_near_ties(seed=0):
    """Groups whose quotients x / s sit a few float32 ulps off an E4M3
    rounding boundary.

    For amax with a short mantissa that is not a multiple of 7, s =
    fl32(amax / 448) is inexact, while x = 21/16 * 2^e * amax / 448 (and
    x = 7 * 2^-10 * amax / 448, a subnormal-range midpoint) is an exact BF16
    value; x / s then lands within the scale's rounding error of the midpoint,
    on the side that error decides.  These are the inputs on which a
    reciprocal-multiply quantiser would disagree with the division."""
    rng = np.random.default_rng(seed)
    rows = []
    for amax_m in range(33, 64, 2):
        if amax_m % 7 == 0:
            continue
        for e0 in (-30, -7, 0, 9, 40):
            amax = float(amax_m) * 2.0 ** (e0 - 5)
            xs = [3.0 * amax * 2.0 ** (e - 10) for e in range(-6, 8)]  # m = 21/16 * 2^e
            xs += [amax * 2.0 ** -16, 3.0 * amax * 2.0 ** -16]          # m = 7 * 2^-10, 21 * 2^-10
            xs = np.array(xs, dtype=np.float64)
            row = np.zeros(128, dtype=np.float32)
            row[0] = amax
            n = len(xs)
            signs = np.where(rng.random(n) < 0.5, -1.0, 1.0)
            row[1:1 + n] = (signs * xs).astype(np.float32)
            row[1 + n:] = (rng.uniform(-1, 1, 127 - n) * amax).astype(np.float32)
            rows.append(row)
    x = np.stack(rows)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(f32(xb)[:, :17], x[:, :17]), "constructed values must be BF16-exact"
    return xb


def test_act_quant_near_ties_inexact_scale():
    x = inexact_scale_near_ties()
    _act_parity(x)
    # the construction really produces quotients off a midpoint by less than 2^-20 relative
    xf = f32(x).astype(np.float64)
    s = oracle.fl32_div(np.max(np.abs(f32(x)), axis=1), np.float32(448.0)).astype(np.float64)
    q = np.abs(xf[:, 1:15] / s[:, None])
    e = np.floor(np.log2(q))
    mant = q / 2.0 ** e  # in [1, 2)
    assert np.all(np.abs(mant - 21 / 16) < 2.0 ** -20 * 21 / 16)


def test_weight_quant_near_ties_inexact_scale():
    rows = f32(inexact_scale_near_ties(seed=1))
    # one 128x128 block per amax: the constructed row first, then rows well below amax
    blocks = []
    rng = np.random.default_rng(2)
    for r in rows[:12]:
        blk = (rng.uniform(-0.5, 0.5, (128, 128)) * float(np.max(np.abs(r)))).astype(np.float32)
        blk[0] = r
        blocks.append(blk)
    w = torch.from_numpy(np.concatenate(blocks, axis=0)).to(torch.bfloat16)
    _weight_parity(w)


def test_act_quant_every_bf16_magnitude():
    """One 1x128 group per positive finite BF16 value (subnormals included):
    the group's amax takes every value a BF16 input can produce, so the
    scale s = fl32(amax / 448) is checked for all of them bit for bit."""
    bits = np.arange(1, 0x7F80, dtype=np.uint32)
    amax = (bits << 16).view(np.float32)
    rng = np.random.default_rng(7)
    x = (rng.uniform(-1.0, 1.0, (len(bits), 128)) * amax[:, None].astype(np.float64)).astype(np.float32)
    x = f32(torch.from_numpy(x).to(torch.bfloat16))          # BF16 rounding never exceeds amax
    pos = rng.integers(0, 128, len(bits))
    sign = np.where(rng.random(len(bits)) < 0.5, -1.0, 1.0).astype(np.float32)
    x[np.arange(len(bits)), pos] = sign * amax
    assert np.array_equal(np.max(np.abs(x), axis=1), amax)
    _act_parity(torch.from_numpy(x).to(torch.bfloat16))


def test_act_quant_all_significand_pairs():
    """Every (amax significand, x significand) pair at every exponent offset
    that gives a non-zero code or the zero boundary, both signs.  amax and x
    are BF16, so s = fl32(amax / 448) has 128 possible significands and this
    covers the quotient x / s exhaustively up to powers of two."""
    sig = 1.0 + np.arange(128) / 128.0
    groups = []
    for a in sig:
        for d in range(-20, 1):
            xs = sig * 2.0 ** d * 4.0
            if d == 0:
                xs = np.where(sig <= a, xs, a * 4.0)  # stay below the group's amax
            for sign in (1.0, -1.0):
                g = np.concatenate([[a * 4.0], sign * xs[:127]])
                groups.append(g)
                groups.append(np.concatenate([[a * 4.0], sign * xs[127:], np.zeros(126)]))
    x = np.asarray(groups, dtype=np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(f32(xb), x), "inputs must be BF16-exact"
    _act_parity(xb)


@pytest.mark.parametrize("M,K", [(4096, 4096)])
def test_act_quant_random_sweep(M, K):
    """16.7M elements with a random power-of-two magnitude per row: every code
    and scale matches the oracle (the FMA-corrected quotient and, for rows
    with scales below 2^-64, the IEEE division)."""
    g = torch.Generator().manual_seed(123)
    x = torch.randn(M, K, generator=g) * torch.pow(2.0, torch.randint(-40, 40, (M, 1), generator=g).float())
    _act_parity(x.to(torch.bfloat16))


def test_weight_quant_random_sweep():
    g = torch.Generator().manual_seed(321)
    w = torch.randn(4096, 4096, generator=g)
    w = w * torch.pow(2.0, torch.randint(-40, 40, (32, 1, 32, 1), generator=g).float()).expand(32, 128, 32, 128).reshape(4096, 4096)
    _weight_parity(w.to(torch.bfloat16))
