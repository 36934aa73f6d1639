"""The GPU quantisers form fl32(x / s) without a division, by Markstein's FMA
correction of the quotient (P. Markstein, "Computation of elementary functions
on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990):

    r = fl32(1 / s)  (correctly rounded)
    q0 = fl32(x r);  e = fl32(x - q0 s)  (one FMA, exact);  q1 = fl32(q0 + e r)  (one FMA)

These CPU tests emulate that chain with exact float32 rounding (float64
intermediates where they are exact, a two-sum where they are not) and check
q1 == fl32(x / s):

- exhaustively over all 128 BF16 significands of x and all 2^23 float32
  significands of s (the chain is invariant under power-of-two scaling while
  it stays in the normal range, so this covers every normal case);
- with scales down to 2^-64, the smallest scale the GPU path sends through
  the chain, and every quotient binade that can give a non-zero E4M3 code;
- and that the checker itself fails when the correction step is dropped or
  the reciprocal is one ulp off (so a pass means something).

Only the quantisers' method is emulated here; the oracle divides.
"""
import numpy as np
import pytest

import oracle

SIG_X = (1.0 + np.arange(128) / 128.0).astype(np.float32)


def _all_scale_significands():
    return (np.arange(1 << 23, dtype=np.uint32) + np.uint32(0x3F800000)).view(np.float32)


def _rn32_exact_sum(a64, b64):
    """fl32(a + b) for float64 a, b whose exact sum may need more than 53
    bits: two-sum, then a float32 rounding that sees the low part when the
    high part sits exactly on a float32 midpoint."""
    hi = a64 + b64
    bv = hi - a64
    lo = (a64 - (hi - bv)) + (b64 - bv)
    c = hi.astype(np.float32)
    bits = hi.view(np.uint64)
    mid = ((bits & np.uint64((1 << 29) - 1)) == np.uint64(1 << 28)) & (lo != 0)
    if mid.any():
        h = hi[mid]
        smaller = (bits[mid] & ~np.uint64((1 << 29) - 1)).view(np.float64).astype(np.float32)  # exact
        larger = np.nextafter(smaller, np.copysign(np.float32(np.inf), h).astype(np.float32))
        c[mid] = np.where((lo[mid] > 0) == (h > 0), larger, smaller)
    return c


def _chain(x, s, r=None, correct=True):
    s64 = s.astype(np.float64)
    if r is None:
        r = (1.0 / s64).astype(np.float32)  # innocuous double rounding: fl32(1 / s)
    q0 = (x * r).astype(np.float32)
    if not correct:
        return q0
    q064 = q0.astype(np.float64)
    e = (x.astype(np.float64) - q064 * s64).astype(np.float32)  # exact difference, one rounding
    er = e.astype(np.float64) * r.astype(np.float64)            # exact: 48 bits
    return _rn32_exact_sum(q064, er)


def _mismatches(xs, s, **kw):
    bad = 0
    s64 = s.astype(np.float64)
    for xv in xs:
        x = np.full(s.shape, xv, dtype=np.float32)
        want = (x.astype(np.float64) / s64).astype(np.float32)  # fl32(x / s), innocuous double rounding
        got = _chain(x, s, **kw)
        bad += int(np.count_nonzero(got.view(np.uint32) != want.view(np.uint32)))
    return bad


def test_two_sum_rounding_helper():
    """_rn32_exact_sum against exact rationals, including sums whose float64
    part is exactly a float32 midpoint."""
    from fractions import Fraction
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.standard_normal(64), [1.0 + 2.0 ** -24, -(1.0 + 2.0 ** -24), 3.0 * 2.0 ** -25] * 2])
    b = np.concatenate([rng.standard_normal(64) * 2.0 ** -40, [2.0 ** -60, 2.0 ** -60, -(2.0 ** -70)],
                        [-(2.0 ** -60), -(2.0 ** -60), 2.0 ** -70]])
    got = _rn32_exact_sum(a, b)
    for i in range(len(a)):
        exact = Fraction(float(a[i])) + Fraction(float(b[i]))
        c0 = np.float32(float(exact))
        cands = [np.nextafter(c0, np.float32(-np.inf)), c0, np.nextafter(c0, np.float32(np.inf))]
        best = min(cands, key=lambda c: (abs(Fraction(float(c)) - exact), int(np.array(c).view(np.uint32)) & 1))
        assert got[i] == best, (a[i], b[i], got[i], best)


def test_correction_exact_over_all_significands():
    s = _all_scale_significands()
    assert _mismatches(SIG_X, s) == 0


def test_correction_exact_at_small_scales():
    """Scales at 2^-64 .. 2^-60 and every quotient binade from 2^-12 (below
    half the smallest E4M3 subnormal) to 2^8."""
    rng = np.random.default_rng(1)
    sig = np.concatenate([rng.integers(0, 1 << 23, 4096), [0, 1, (1 << 23) - 1]]).astype(np.uint32)
    base = (sig + np.uint32(0x3F800000)).view(np.float32).astype(np.float64)
    for es in (-64, -62, -60):
        s = (base * 2.0 ** es).astype(np.float32)
        for qb in range(-12, 9):
            xs = (SIG_X.astype(np.float64) * 2.0 ** (es + qb)).astype(np.float32)
            assert _mismatches(xs, s) == 0, (es, qb)


def test_checker_catches_planted_mistakes():
    s = _all_scale_significands()
    assert _mismatches(SIG_X[::8], s[::64], correct=False) > 0
    r_off = np.nextafter((1.0 / s.astype(np.float64)).astype(np.float32), np.float32(0))
    assert _mismatches(np.float32([1.75, 1.875]), s, r=r_off) > 0


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_codes_through_the_chain_match_the_oracle(sign):
    """End to end on the quantiser's own domain: every BF16 amax significand
    and x significand, quotient binades down to the zero boundary, coded with
    the oracle's E4M3 encoder -- identical to the oracle's quantisation."""
    groups = []
    for a in SIG_X.astype(np.float64):
        for d in range(-20, 1):
            xs = SIG_X.astype(np.float64) * 2.0 ** d
            if d == 0:
                xs = np.where(SIG_X <= a, xs, a)
            groups.append(np.concatenate([[a], sign * xs[:127]]))
    x = np.asarray(groups, dtype=np.float32)
    q_ref, s_ref = oracle.quant_act_1x128(x)
    s = s_ref[0]                                    # [M] scales of the single K block
    q1 = _chain(x, np.repeat(s[:, None], 128, axis=1).astype(np.float32))
    codes = oracle.e4m3_encode_rne_satfinite(q1)
    assert np.array_equal(codes, q_ref)
