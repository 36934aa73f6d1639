"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each ``pin_*`` function takes an oracle module ``o`` and raises
AssertionError when the oracle disagrees with the fact it checks.  The
oracle's own tests call them with the real oracle; the mutation tests call
them with copies of the oracle that carry a planted mistake and expect at
least one pin to fail.

What the pins rest on:
  * the E4M3FN format (OCP OFP8 spec rev 1.0, Table 1), through fixed code
    points, an exhaustive code round trip and tie-breaking at every midpoint;
  * an independent library routine, torch's float8_e4m3fn cast, in the range
    where it and the method agree (|v| <= 448, no saturation involved);
  * exact rational arithmetic (fractions.Fraction) for divisions, scales and a
    brute-force GEMM on tiny inputs;
  * closed forms and invariants of the method: the amax element maps to
    +-448, scaling a group by 2**j leaves its codes unchanged, a group's
    codes depend only on that group, constant operands give a closed-form
    product, one-hot weights select dequantised activation columns, and the
    product is linear under power-of-two scaling.
The method itself is the one of "The Definitive Information To Deepseek"
(paragraph 3, "Figure 7 (a)": 1x128 activation tiles, 128x128 weight
blocks; paragraph 2: online per-group scaling; paragraph 4: FP8 GEMM with
BF16 output; paragraph 1: promotion of partial sums).
"""

from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _nearest_f32(q: Fraction) -> np.float32:
    """Correctly rounded float32 of an exact rational (ties to even), found by
    bracketing with neighbouring float32 values and comparing exactly."""
    approx = np.float32(float(q))  # within an ulp or two
    cands = set()
    c = approx
    for _ in range(3):
        c = np.nextafter(c, np.float32(-np.inf), dtype=np.float32)
    for _ in range(7):
        cands.add(c)
        c = np.nextafter(c, np.float32(np.inf), dtype=np.float32)
    best = None
    for c in sorted(cands, key=float):
        if not np.isfinite(c):
            continue
        d = abs(Fraction(float(c)) - q)
        if best is None or d < best[0] or (d == best[0] and (c.view(np.uint32) & 1) == 0):
            best = (d, c)
    return best[1]


def _frac_dec(code: int) -> Fraction:
    s = -1 if code & 0x80 else 1
    e = (code >> 3) & 0xF
    m = code & 7
    if e == 0:
        return s * Fraction(m, 8) * Fraction(1, 64)
    return s * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


# ---------------------------------------------------------------------------
# E4M3 codec
# ---------------------------------------------------------------------------

def pin_codec_format_points(o):
    for code, value in _read_table("e4m3_format_points.txt"):
        c = int(code, 16)
        v = float(value)
        got = float(o.e4m3_decode(np.array([c], dtype=np.uint8))[0])
        assert got == v, f"decode 0x{c:02X}: {got} != {v}"
        enc = int(o.e4m3_encode_rne_satfinite(np.array([v], dtype=np.float32))[0])
        if v == 0.0:
            continue  # +0 / -0 handled by pin_codec_sign_of_zero
        assert enc == c, f"encode {v}: 0x{enc:02X} != 0x{c:02X}"
    nan = o.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))
    assert np.all(np.isnan(nan)), "0x7F/0xFF must decode to NaN"


def pin_codec_roundtrip(o):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = o.e4m3_decode(codes)
    assert np.all(np.isfinite(vals))
    back = o.e4m3_encode_rne_satfinite(vals.astype(np.float32))
    assert np.array_equal(back, codes), "decode -> encode must reproduce all 254 finite codes"
    pos = vals[: 0x7F]
    assert np.all(np.diff(pos) > 0), "positive codes must increase in value"


def pin_codec_ties(o):
    """Exact midpoints between neighbours go to the even code; one float32 ulp
    either side goes to the nearer neighbour.  Both signs."""
    pos = o.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    for c in range(0x7E):
        lo, hi = pos[c], pos[c + 1]
        mid = np.float32((lo + hi) / 2)  # exact: E4M3 midpoints fit in float32
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        up = np.nextafter(mid, np.float32(np.inf), dtype=np.float32)
        dn = np.nextafter(mid, np.float32(-np.inf), dtype=np.float32)
        for sgn, sbit in ((1, 0), (-1, 0x80)):
            got = o.e4m3_encode_rne_satfinite(np.array([sgn * mid, sgn * up, sgn * dn], dtype=np.float32))
            assert int(got[0]) == (even | sbit), f"tie at {sgn * mid} -> 0x{int(got[0]):02X}"
            assert int(got[1]) == ((c + 1) | sbit), f"above tie {sgn * up} -> 0x{int(got[1]):02X}"
            assert int(got[2]) == (c | sbit), f"below tie {sgn * dn} -> 0x{int(got[2]):02X}"


def pin_codec_saturation(o):
    big = np.array([448.0, 448.5, 463.99, 464.0, 464.01, 479.9, 480.0, 512.0, 1e6, 3.0e38], dtype=np.float32)
    got = o.e4m3_encode_rne_satfinite(np.concatenate([big, -big]))
    assert np.all(got[: len(big)] == 0x7E), got
    assert np.all(got[len(big):] == 0xFE), got


def pin_codec_sign_of_zero(o):
    v = np.array([0.0, -0.0, -(2.0 ** -11), -(2.0 ** -10), 2.0 ** -11, -1e-30], dtype=np.float32)
    got = o.e4m3_encode_rne_satfinite(v)
    assert list(got) == [0x00, 0x80, 0x80, 0x80, 0x00, 0x80], [hex(int(g)) for g in got]


def structured_f32_patterns(low_bits_random=4, seed=1234):
    """float32 bit patterns with |v| <= 448: every exponent, every value of the
    top 12 mantissa bits, and for the low 11 bits the edge patterns plus a few
    random ones.  E4M3 rounding boundaries all sit at mantissa bit 19 or
    above, so this covers every round/sticky combination that matters."""
    rng = np.random.default_rng(seed)
    low = [0x000, 0x001, 0x002, 0x3FF, 0x400, 0x401, 0x7FE, 0x7FF]
    low += list(rng.integers(0, 0x800, size=low_bits_random))
    exps = np.arange(0, 136, dtype=np.uint32)          # biased exponent up to 2^8
    top = np.arange(0, 1 << 12, dtype=np.uint32)
    base = (exps[:, None] << 23) | (top[None, :] << 11)
    bits = (base[:, :, None] | np.array(low, dtype=np.uint32)[None, None, :]).ravel()
    v = bits.view(np.float32)
    v = v[np.abs(v) <= 448.0]
    return np.concatenate([v, -v])


def pin_codec_vs_torch(o, low_bits_random=4):
    import torch

    v = structured_f32_patterns(low_bits_random)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = o.e4m3_encode_rne_satfinite(v)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (
        f"{bad.size} mismatches vs torch float8_e4m3fn, e.g. v={v[bad[:4]]} "
        f"got={got[bad[:4]]} torch={ref[bad[:4]]}")


# ---------------------------------------------------------------------------
# Rounded division and scales
# ---------------------------------------------------------------------------

def _division_samples(seed=7, n=3000):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(n).astype(np.float32) * np.float32(2.0) ** rng.integers(-30, 30, n).astype(np.float32)
    b = np.abs(rng.standard_normal(n).astype(np.float32)) * np.float32(2.0) ** rng.integers(-30, 30, n).astype(np.float32)
    # edge cases: subnormal divisors / quotients, exact quotients, 448 itself
    a = np.concatenate([a, np.array([448, 1, 3, 2.0 ** -140, 56, 1e-38, 2.0 ** -120], dtype=np.float32)])
    b = np.concatenate([b, np.array([448, 448, 448, 448, 0.125, 448, 2.0 ** -130], dtype=np.float32)])
    return a, b


def pin_fl32_div_exact(o):
    a, b = _division_samples()
    got = o.fl32_div(a, b)
    for ai, bi, gi in zip(a, b, got):
        want = _nearest_f32(Fraction(float(ai)) / Fraction(float(bi)))
        assert gi.view(np.uint32) == want.view(np.uint32), f"fl32({ai}/{bi}) = {gi} != {want}"


def pin_scale_definition(o):
    """s is exactly the float32 nearest to amax / 448 (checked with rationals),
    for ordinary, tiny (subnormal-scale) and large groups."""
    rng = np.random.default_rng(11)
    rows = []
    for e in (-140, -126, -120, -60, -3, 0, 5, 60, 120):
        r = (rng.standard_normal(128) * 2.0 ** e).astype(np.float32)
        rows.append(r)
    x = np.stack(rows)
    _, sa = o.quant_act_1x128(x)
    for m in range(x.shape[0]):
        amax = Fraction(float(np.max(np.abs(x[m]))))
        want = _nearest_f32(amax / 448)
        assert sa[0, m].view(np.uint32) == want.view(np.uint32), f"row {m}: s={sa[0, m]} != {want}"


# ---------------------------------------------------------------------------
# Quantisation
# ---------------------------------------------------------------------------

def pin_quant_worked_example(o):
    rows = _read_table("quant_worked_example.txt")
    x = np.zeros((1, 256), dtype=np.float32)
    want = np.zeros(128, dtype=np.uint8)
    scale = None
    for r in rows:
        if r[0] == "scale":
            scale = float(r[1])
            continue
        i, xv, _, code = int(r[0]), float(r[1]), r[2], int(r[3], 16)
        x[0, i] = np.float32(xv)
        want[i] = code
    # second group all zeros, with a negative zero in it
    x[0, 130] = -0.0
    qa, sa = o.quant_act_1x128(x)
    assert np.array_equal(qa[0, :128], want), [hex(int(c)) for c in qa[0, :13]]
    assert float(sa[0, 0]) == scale
    assert float(sa[1, 0]) == 0.0 and np.all(qa[0, 128:] == 0), "all-zero group: s = 0, codes 0x00"


def exact_tie_groups(scales=(1.5, 1.75, 1.25, 1.3125, 1.171875, 0.75 * 2.0 ** -20, 1.5 * 2.0 ** 30)):
    """Groups whose quotients x / s are exact E4M3 midpoints.

    For each scale s (short mantissa, so every product below is exact in
    float32) the group holds the amax 448 * s first, then m * s for the
    midpoints m between neighbouring codes, alternating signs.  Returns
    (x float32 [len(scales), 128*ceil(n/127)], expected codes uint8)."""
    pos = [float(_frac_dec(c)) for c in range(0x7F)]
    mids = [((pos[c] + pos[c + 1]) / 2, c if c % 2 == 0 else c + 1) for c in range(0x7E)]
    per_row = [(448.0, 0x7E)] + mids  # 127 entries
    width = 128
    xs, codes = [], []
    for s in scales:
        row = np.zeros(width, dtype=np.float32)
        crow = np.zeros(width, dtype=np.uint8)
        for i, (m, c) in enumerate(per_row):
            sign = -1.0 if (i % 2) else 1.0
            row[i] = np.float32(sign * m * s)
            assert float(row[i]) == sign * m * s
            crow[i] = c | (0x80 if sign < 0 else 0)
        xs.append(row)
        codes.append(crow)
    return np.stack(xs), np.stack(codes)


def pin_quant_exact_ties(o):
    """Exact midpoint quotients must round to the even code, which only a
    correctly rounded x / s guarantees (x * fl32(1/s) can land an ulp off)."""
    x, want = exact_tie_groups()
    qa, sa = o.quant_act_1x128(x)
    bad = np.nonzero(qa != want)
    assert bad[0].size == 0, f"{bad[0].size} tie codes wrong, e.g. row {bad[0][:3]} col {bad[1][:3]}"


def pin_amax_maps_to_448(o):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 512)).astype(np.float32)
    x *= (2.0 ** rng.integers(-110, 100, size=(64, 1))).astype(np.float32)
    qa, sa = o.quant_act_1x128(x)
    g = np.abs(x.reshape(64, 4, 128))
    idx = np.argmax(g, axis=2)
    codes = qa.reshape(64, 4, 128)
    for m in range(64):
        for kb in range(4):
            c = int(codes[m, kb, idx[m, kb]])
            assert c in (0x7E, 0xFE), f"amax element of group ({m},{kb}) -> 0x{c:02X}"


def pin_quant_error_bound(o):
    """|dec(q) * s - x| <= half an E4M3 ulp of x/s, times s, with a float32
    rounding allowance (x/s itself is rounded to float32 first)."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((32, 384)) * 3).astype(np.float32)
    qa, sa = o.quant_act_1x128(x)
    s = np.repeat(sa.T.astype(np.float64), 128, axis=1)
    v = x.astype(np.float64) / s
    a = np.abs(v)
    # E4M3 spacing around |v|: 2^(e-3) for normals (e = floor(log2 a)), 2^-9 below 2^-6
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    ulp = np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))
    err = np.abs(o.e4m3_decode(qa) * s - x)
    assert np.all(err <= 0.5 * ulp * s * (1 + 2.0 ** -22) + 1e-300)


def pin_quant_pow2_invariance(o):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((8, 256)).astype(np.float32)
    q0, s0 = o.quant_act_1x128(x)
    for j in (-20, -3, 1, 7, 40):
        q1, s1 = o.quant_act_1x128((x * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(q0, q1), f"codes changed under 2^{j} scaling"
        assert np.array_equal(s1, (s0 * np.float32(2.0 ** j)).astype(np.float32))
    w = (rng.standard_normal((256, 256)) * 0.02).astype(np.float32)
    qw0, sw0 = o.quant_weight_128x128(w)
    qw1, sw1 = o.quant_weight_128x128((w * np.float32(8.0)).astype(np.float32))
    assert np.array_equal(qw0, qw1) and np.array_equal(sw1, sw0 * np.float32(8.0))


def pin_quant_locality(o):
    """Changing one element changes only its own group's scale and codes."""
    rng = np.random.default_rng(13)
    x = rng.standard_normal((6, 512)).astype(np.float32)
    qa, sa = o.quant_act_1x128(x)
    x2 = x.copy()
    x2[4, 300] = 1000.0  # row 4, group kb=2
    qb, sb = o.quant_act_1x128(x2)
    diff_groups = {(m, k // 128) for m, k in zip(*np.nonzero(qa != qb))}
    assert diff_groups == {(4, 2)}, diff_groups
    ds = {(kb, m) for kb, m in zip(*np.nonzero(sa != sb))}
    assert ds == {(2, 4)}, ds
    assert sa.shape == (4, 6)

    w = (rng.standard_normal((384, 512)) * 0.02).astype(np.float32)
    qw, sw = o.quant_weight_128x128(w)
    w2 = w.copy()
    w2[200, 70] = 5.0  # block (nb=1, kb=0)
    qw2, sw2 = o.quant_weight_128x128(w2)
    blocks = {(n // 128, k // 128) for n, k in zip(*np.nonzero(qw != qw2))}
    assert blocks == {(1, 0)}, blocks
    assert {(a, b) for a, b in zip(*np.nonzero(sw != sw2))} == {(1, 0)}
    assert sw.shape == (3, 4)


def pin_weight_structure(o):
    # block-constant magnitudes with random signs: every code +-0x7E and
    # sw[nb, kb] = fl32(c / 448) for the block's constant c
    rng = np.random.default_rng(17)
    NB, KB = 3, 2
    c = (2.0 ** rng.integers(-8, 8, size=(NB, KB))).astype(np.float32) * np.float32(1.5)
    sign = np.where(rng.random((NB * 128, KB * 128)) < 0.5, -1.0, 1.0).astype(np.float32)
    w = np.repeat(np.repeat(c, 128, 0), 128, 1) * sign
    qw, sw = o.quant_weight_128x128(w)
    assert np.all((qw == 0x7E) | (qw == 0xFE))
    assert np.array_equal((qw == 0xFE), sign < 0)
    for nb in range(NB):
        for kb in range(KB):
            want = _nearest_f32(Fraction(float(c[nb, kb])) / 448)
            assert sw[nb, kb] == want
    # 128x128 blocks are symmetric under transposition
    w = (rng.standard_normal((256, 384)) * 0.02).astype(np.float32)
    qw, sw = o.quant_weight_128x128(w)
    qt, st = o.quant_weight_128x128(np.ascontiguousarray(w.T))
    assert np.array_equal(qt, qw.T) and np.array_equal(st, sw.T)


# ---------------------------------------------------------------------------
# GEMM
# ---------------------------------------------------------------------------

def pin_gemm_bruteforce(o):
    """Element-by-element exact rational sum on tiny inputs: the scale of
    element (m, k) is sa[k//128, m], of weight (n, k) is sw[n//128, k//128],
    and each 128-wide chunk is summed exactly before scaling."""
    rng = np.random.default_rng(21)
    for M, N, K in ((3, 128, 128), (2, 256, 256), (4, 128, 384)):
        x = rng.standard_normal((M, K)).astype(np.float32)
        w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        qa, sa = o.quant_act_1x128(x)
        qw, sw = o.quant_weight_128x128(w)
        y = o.blockscaled_gemm(qa, sa, qw, sw)
        assert y.shape == (M, N)
        dec = [_frac_dec(c) for c in range(256)]
        ncheck = [0, 1, N // 2 + 3, N - 1]
        for m in range(M):
            for n in ncheck:
                tot = Fraction(0)
                mag = Fraction(0)
                for kb in range(K // 128):
                    part = sum(dec[int(qa[m, k])] * dec[int(qw[n, k])] for k in range(kb * 128, kb * 128 + 128))
                    term = Fraction(float(sa[kb, m])) * Fraction(float(sw[n // 128, kb])) * part
                    tot += term
                    mag += abs(term)
                # float64 may round each scaled chunk and each addition: a few
                # units of 2^-53 relative to the sum of |terms|
                bound = 4 * len(range(K // 128)) * 2.0 ** -53 * float(mag)
                assert abs(Fraction(float(y[m, n])) - tot) <= Fraction(bound), (M, N, K, m, n, y[m, n], float(tot))


def pin_gemm_closed_form(o):
    """X = a everywhere and W = b everywhere: every code is 0x7E, so
    Y = K * (448 s_x) * (448 s_w) exactly."""
    for a, b, K in ((1.0, 0.5, 256), (3.0, -0.0078125, 512), (0.1, 7.0, 128)):
        x = np.full((5, K), np.float32(a), dtype=np.float32)
        w = np.full((256, K), np.float32(b), dtype=np.float32)
        qa, sa = o.quant_act_1x128(x)
        qw, sw = o.quant_weight_128x128(w)
        y = o.blockscaled_gemm(qa, sa, qw, sw)
        sx = float(sa[0, 0])
        sw0 = float(sw[0, 0])
        want = K * (448.0 * sx) * (448.0 * sw0)
        if b < 0:
            want = -want
        assert np.all(y == want), (a, b, K, y[0, 0], want)


def pin_gemm_onehot(o):
    """W[n, k] = 448 if k == perm[n] else 0: s_w = 1 for blocks that hold a 448
    and 0 elsewhere, so Y[m, n] = 448 * dequantised X[m, perm[n]]."""
    rng = np.random.default_rng(23)
    M, N, K = 7, 256, 384
    x = rng.standard_normal((M, K)).astype(np.float32)
    perm = rng.permutation(K)[:N]
    w = np.zeros((N, K), dtype=np.float32)
    w[np.arange(N), perm] = 448.0
    qa, sa = o.quant_act_1x128(x)
    qw, sw = o.quant_weight_128x128(w)
    y = o.blockscaled_gemm(qa, sa, qw, sw)
    xdq = o.e4m3_decode(qa) * np.repeat(sa.T.astype(np.float64), 128, axis=1)
    assert np.array_equal(y, 448.0 * xdq[:, perm])


def pin_gemm_linearity(o):
    rng = np.random.default_rng(29)
    x = rng.standard_normal((9, 256)).astype(np.float32)
    w = (rng.standard_normal((128, 256)) * 0.02).astype(np.float32)
    y0, _ = o.linear_forward(x, w)
    for j in (-5, 3, 12):
        y1, _ = o.linear_forward((x * np.float32(2.0 ** j)).astype(np.float32), w)
        assert np.array_equal(y1, y0 * 2.0 ** j)


def pin_gemm_rows_columns(o):
    """Row m of Y depends only on row m of X, column n only on row n of W."""
    rng = np.random.default_rng(31)
    x = rng.standard_normal((5, 256)).astype(np.float32)
    w = (rng.standard_normal((256, 256)) * 0.02).astype(np.float32)
    y0, _ = o.linear_forward(x, w)
    x2 = x.copy()
    x2[3] *= -2.5
    y1, _ = o.linear_forward(x2, w)
    changed = np.nonzero(np.any(y0 != y1, axis=1))[0]
    assert list(changed) == [3], changed


def pin_grouped(o):
    rng = np.random.default_rng(37)
    G, N, K = 5, 128, 256
    counts = [3, 0, 130, 1, 0]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    x = rng.standard_normal((int(offsets[-1]), K)).astype(np.float32)
    w = (rng.standard_normal((G, N, K)) * 0.02).astype(np.float32)
    qa, sa = o.quant_act_1x128(x)
    qws, sws = zip(*(o.quant_weight_128x128(w[g]) for g in range(G)))
    qw, sw = np.stack(qws), np.stack(sws)
    y = o.blockscaled_grouped_gemm(offsets, qa, sa, qw, sw)
    assert y.shape == (offsets[-1], N)
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 > r0:
            ref = o.blockscaled_gemm(qa[r0:r1], sa[:, r0:r1], qw[g], sw[g])
            assert np.array_equal(y[r0:r1], ref), g
    # one group equals the dense product
    yd = o.blockscaled_gemm(qa, sa, qw[2], sw[2])
    y1 = o.blockscaled_grouped_gemm([0, offsets[-1]], qa, sa, qw[2:3], sw[2:3])
    assert np.array_equal(y1, yd)
    # stacked weight quantisation equals per-group quantisation (N % 128 == 0)
    qst, sst = o.quant_weight_128x128(w.reshape(G * N, K))
    assert np.array_equal(qst.reshape(G, N, K), qw) and np.array_equal(sst.reshape(G, N // 128, K // 128), sw)


# ---------------------------------------------------------------------------
# Block dequantisation (FP8 -> BF16 weights)
# ---------------------------------------------------------------------------

def pin_bf16_round(o):
    """Round-to-nearest-even BF16 against torch's float32 -> bfloat16 cast
    (an independent library routine) on structured bit patterns: every
    exponent, and low halves at and around the rounding midpoint 0x8000."""
    import torch

    exps = np.arange(1, 255, dtype=np.uint32)
    hi = np.array([0x000, 0x001, 0x07E, 0x07F, 0x040, 0x041], dtype=np.uint32)
    lo = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    bits = ((exps[:, None, None] << 23) | (hi[None, :, None] << 16) | lo[None, None, :]).ravel()
    v = bits.view(np.float32)
    v = np.concatenate([v, -v, np.array([0.0, -0.0], dtype=np.float32)])
    v = v[np.isfinite(v) & (np.abs(v) < 3.3e38)]
    want = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    got = o.bf16_round(v)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def pin_dequant_roundtrip(o):
    """dequant(quant(W)) reproduces W to within half an E4M3 ulp of the block
    (times its scale) plus the BF16 rounding; codes 0x7E with s = 1.5 give
    exactly 672; an all-zero block gives zeros."""
    rng = np.random.default_rng(41)
    w = (rng.standard_normal((256, 384)) * 0.02).astype(np.float32)
    w[128:256, 0:128] = 0.0
    qw, sw = o.quant_weight_128x128(w)
    y = o.dequant_weight_128x128_bf16(qw, sw).astype(np.float64)
    s = np.repeat(np.repeat(sw.astype(np.float64), 128, 0), 128, 1)
    v = np.abs(w.astype(np.float64)) / np.where(s > 0, s, 1)
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
    ulp = np.where(v < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))
    bound = 0.5 * ulp * s * (1 + 2.0 ** -20) + np.abs(w) * 2.0 ** -8 + 1e-300
    assert np.all(np.abs(y - w) <= bound)
    assert np.all(y[128:256, 0:128] == 0.0)
    q = np.full((128, 128), 0x7E, dtype=np.uint8)
    assert np.all(o.dequant_weight_128x128_bf16(q, np.array([[1.5]], dtype=np.float32)) == 672.0)
    # the float32 product is rounded to BF16 once more: 0x39 (1.125) * 1.0078125 = 1.1337890625 -> 1.1328125
    q = np.full((128, 128), 0x39, dtype=np.uint8)
    got = o.dequant_weight_128x128_bf16(q, np.array([[1.0078125]], dtype=np.float32))
    assert np.all(got == np.float32(1.1328125)), got[0, 0]


def pin_dequant_float64(o):
    """The float64 block dequantisation dec(q) * s on a hand-built 256 x 384
    matrix of six blocks with six different scales: sampled elements equal
    the exact rational product of the code's value (from the E4M3 format)
    and its own block's scale, so a transposed, reversed or mis-broadcast
    scale fails; and its float32 rounding, rounded to BF16, is exactly the
    BF16 dequantisation (the float64 product of a <= 4-bit code value and a
    float32 scale is exact)."""
    rng = np.random.default_rng(47)
    codes = rng.integers(0, 256, size=(256, 384)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x7E  # NaN codes are outside the contract
    sw = np.array([[1.5, 2.0 ** -3, 3.0], [0.75, 5.0, 2.0 ** -10]], dtype=np.float32)
    y = o.dequant_weight_128x128(codes, sw)
    assert y.shape == (256, 384) and y.dtype == np.float64
    pos = [(0, 0), (127, 127), (128, 0), (0, 128), (255, 383), (129, 257), (5, 300), (200, 140)]
    pos += [tuple(p) for p in rng.integers(0, [256, 384], size=(200, 2))]
    for n, k in pos:
        want = _frac_dec(int(codes[n, k])) * Fraction(float(sw[n // 128, k // 128]))
        assert Fraction(float(y[n, k])) == want, (n, k, y[n, k], float(want))
    y16 = o.dequant_weight_128x128_bf16(codes, sw)
    assert np.array_equal(o.bf16_round(y.astype(np.float32)).view(np.uint32), y16.view(np.uint32))


# ---------------------------------------------------------------------------
# Backward GEMMs
# ---------------------------------------------------------------------------

def pin_rowscaled_bruteforce(o):
    """Exact rational sum on tiny inputs: element (m, n) gets
    sa[kb, m] * sb[kb, n] times the exact chunk sum, per 128-wide chunk."""
    rng = np.random.default_rng(43)
    dec = [_frac_dec(c) for c in range(256)]
    for M, N, K in ((3, 5, 128), (2, 4, 256)):
        a = rng.standard_normal((M, K)).astype(np.float32)
        b = (rng.standard_normal((N, K)) * 0.1).astype(np.float32)
        qa, sa = o.quant_act_1x128(a)
        qb, sb = o.quant_act_1x128(b)
        y = o.blockscaled_gemm_rowscaled(qa, sa, qb, sb)
        assert y.shape == (M, N)
        for m in range(M):
            for n in range(N):
                tot, mag = Fraction(0), Fraction(0)
                for kb in range(K // 128):
                    part = sum(dec[int(qa[m, k])] * dec[int(qb[n, k])] for k in range(kb * 128, kb * 128 + 128))
                    term = Fraction(float(sa[kb, m])) * Fraction(float(sb[kb, n])) * part
                    tot += term
                    mag += abs(term)
                bound = 4 * (K // 128) * 2.0 ** -53 * float(mag)
                assert abs(Fraction(float(y[m, n])) - tot) <= Fraction(bound), (M, N, K, m, n)


def pin_rowscaled_reduces_to_blockscaled(o):
    """With per-column scales that are constant over each 128-wide block of
    output columns, the row-scaled product is the block-scaled one."""
    rng = np.random.default_rng(47)
    x = rng.standard_normal((7, 384)).astype(np.float32)
    w = (rng.standard_normal((256, 384)) * 0.02).astype(np.float32)
    qa, sa = o.quant_act_1x128(x)
    qw, sw = o.quant_weight_128x128(w)
    sb = np.repeat(sw.T, 128, axis=1)  # [K/128, N]: scale of column n in chunk kb = sw[n // 128, kb]
    assert np.array_equal(o.blockscaled_gemm_rowscaled(qa, sa, qw, sb), o.blockscaled_gemm(qa, sa, qw, sw))


def pin_transposed_quant_structure(o):
    """1x128 tiles of x^T are runs of 128 rows of one column of x: constant
    columns code to +-448 with s = fl32(|c| / 448); perturbing one element
    changes only its own (row run, column) group."""
    rng = np.random.default_rng(53)
    c = (rng.standard_normal(6) * 4).astype(np.float32)
    x = np.tile(c, (256, 1))
    q, s = o.quant_act_1x128_t(x)
    assert q.shape == (6, 256) and s.shape == (2, 6)
    assert np.all((q == 0x7E) | (q == 0xFE))
    assert np.array_equal(q == 0xFE, np.tile((c < 0)[:, None], (1, 256)))
    for k in range(6):
        want = _nearest_f32(Fraction(float(abs(c[k]))) / 448)
        assert s[0, k] == want and s[1, k] == want
    x = rng.standard_normal((256, 5)).astype(np.float32)
    q0, s0 = o.quant_act_1x128_t(x)
    x2 = x.copy()
    x2[200, 3] = 100.0
    q1, s1 = o.quant_act_1x128_t(x2)
    assert {(k, m // 128) for k, m in zip(*np.nonzero(q0 != q1))} == {(3, 1)}
    assert {(mb, k) for mb, k in zip(*np.nonzero(s0 != s1))} == {(1, 3)}


def pin_backward_error_bound(o):
    """dX and dW stay within the worst case that E4M3 rounding allows of the
    unquantised float64 products dY . W and dY^T . X (half an E4M3 ulp per
    operand: 2^-4 relative in the normal range, 2^-10 * s below it); a
    transposed or mis-scaled operand breaks the bound by orders of
    magnitude."""
    rng = np.random.default_rng(59)
    M, N, K = 256, 256, 384
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    dy = (rng.standard_normal((M, N)) * 0.5).astype(np.float32)
    dx, dw = o.linear_backward(x, w, dy)

    def err(v, s):
        return np.maximum(np.abs(v) * 2.0 ** -4, s * 2.0 ** -10)

    # dX = dY . W: dY groups 1x128 along N, W blocks 128x128
    _, sdy = o.quant_act_1x128(dy)
    _, sw = o.quant_weight_128x128(w)
    e_dy = err(dy.astype(np.float64), np.repeat(sdy.T.astype(np.float64), 128, axis=1))
    e_w = err(w.astype(np.float64), np.repeat(np.repeat(sw.astype(np.float64), 128, 0), 128, 1))
    ad, aw = np.abs(dy.astype(np.float64)), np.abs(w.astype(np.float64))
    bound = ad @ e_w + e_dy @ aw + e_dy @ e_w
    assert np.all(np.abs(dx - dy.astype(np.float64) @ w.astype(np.float64)) <= bound * (1 + 1e-9) + 1e-30)
    # dW = dY^T . X: both grouped along M
    _, sdyt = o.quant_act_1x128_t(dy)
    _, sxt = o.quant_act_1x128_t(x)
    e_dyt = err(dy.T.astype(np.float64), np.repeat(sdyt.T.astype(np.float64), 128, axis=1))
    e_xt = err(x.T.astype(np.float64), np.repeat(sxt.T.astype(np.float64), 128, axis=1))
    adt, axt = np.abs(dy.T.astype(np.float64)), np.abs(x.T.astype(np.float64))
    bound = adt @ e_xt.T + e_dyt @ axt.T + e_dyt @ e_xt.T
    assert np.all(np.abs(dw - dy.T.astype(np.float64) @ x.astype(np.float64)) <= bound * (1 + 1e-9) + 1e-30)


def pin_backward_linearity(o):
    rng = np.random.default_rng(61)
    x = rng.standard_normal((128, 256)).astype(np.float32)
    w = (rng.standard_normal((128, 256)) * 0.02).astype(np.float32)
    dy = rng.standard_normal((128, 128)).astype(np.float32)
    dx0, dw0 = o.linear_backward(x, w, dy)
    for j in (-6, 5):
        dx1, dw1 = o.linear_backward(x, w, (dy * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(dx1, dx0 * 2.0 ** j) and np.array_equal(dw1, dw0 * 2.0 ** j)


# ---------------------------------------------------------------------------
# Quantisation variants: per token, per channel, E5M6, SwiGLU + 1x128
# ---------------------------------------------------------------------------

def pin_e5m6_format(o):
    """Every finite E5M6 code decodes to the FP16 value whose bit pattern is
    the code shifted left by 4 (an E5M6 number is an FP16 number with the low
    four mantissa bits zero: same sign, bias-15 exponent and subnormal
    rule), checked against numpy's float16; 0x7C0 / 0x7C1 are inf / NaN."""
    codes = np.array([c for c in range(4096) if ((c >> 6) & 0x1F) != 31], dtype=np.uint16)
    want = (codes.astype(np.uint16) << 4).view(np.float16).astype(np.float64)
    got = o.e5m6_decode(codes)
    assert np.array_equal(got, want)
    special = o.e5m6_decode(np.array([0x7C0, 0x7C1, 0xFC0], dtype=np.uint16))
    assert np.isinf(special[0]) and np.isnan(special[1]) and special[2] == -np.inf
    assert o.E5M6_MAX == 65024.0 and float(o.e5m6_decode(np.array([0x7BF], dtype=np.uint16))[0]) == 65024.0


def pin_e5m6_roundtrip_and_ties(o):
    codes = np.array([c for c in range(4096) if ((c >> 6) & 0x1F) != 31], dtype=np.uint16)
    vals = o.e5m6_decode(codes)
    assert np.array_equal(o.e5m6_encode_rne_satfinite(vals.astype(np.float32)), codes)
    pos = o.e5m6_decode(np.arange(31 << 6, dtype=np.uint16))
    assert np.all(np.diff(pos) > 0)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)  # exact in float32
    even = np.where(np.arange(len(mids)) % 2 == 0, np.arange(len(mids)), np.arange(len(mids)) + 1)
    for sgn, sbit in ((1, 0), (-1, 0x800)):
        got = o.e5m6_encode_rne_satfinite(sgn * mids)
        assert np.array_equal(got.astype(np.int64), even | sbit)
        up = np.nextafter(sgn * mids, np.float32(sgn * np.inf), dtype=np.float32)
        assert np.array_equal(o.e5m6_encode_rne_satfinite(up).astype(np.int64), (np.arange(len(mids)) + 1) | sbit)
    big = np.array([65024.0, 65279.0, 65280.0, 70000.0, 3e38], dtype=np.float32)
    assert np.all(o.e5m6_encode_rne_satfinite(big) == 0x7BF) and np.all(o.e5m6_encode_rne_satfinite(-big) == 0xFBF)
    assert list(o.e5m6_encode_rne_satfinite(np.array([0.0, -0.0, -1e-30], dtype=np.float32))) == [0, 0x800, 0x800]


def pin_per_token_and_channel(o):
    """Per-token groups are whole rows, per-channel groups whole columns:
    constant rows / columns code to +-448 with s = fl32(|c| / 448); per
    channel equals per token of the transpose; one element changes only its
    own row's (column's) scale and codes."""
    rng = np.random.default_rng(67)
    c = (rng.standard_normal(5) * 3).astype(np.float32)
    q, s = o.quant_per_token(np.tile(c[:, None], (1, 300)))
    assert q.shape == (5, 300) and s.shape == (5,)
    assert np.all((q == 0x7E) | (q == 0xFE))
    for i in range(5):
        assert s[i] == _nearest_f32(Fraction(float(abs(c[i]))) / 448)
    x = rng.standard_normal((40, 300)).astype(np.float32)
    qc, sc = o.quant_per_channel(x)
    qt, st = o.quant_per_token(np.ascontiguousarray(x.T))
    assert np.array_equal(qc, qt.T) and np.array_equal(sc, st) and sc.shape == (300,)
    amax_col = np.argmax(np.abs(x), axis=0)
    assert np.all(np.isin(qc[amax_col, np.arange(300)], (0x7E, 0xFE)))
    x2 = x.copy()
    x2[7, 11] = 1000.0
    q0, s0 = o.quant_per_token(x)
    q1, s1 = o.quant_per_token(x2)
    assert set(np.nonzero(q0 != q1)[0]) == {7} and set(np.nonzero(s0 != s1)[0]) == {7}
    q0, s0 = o.quant_per_channel(x)
    q1, s1 = o.quant_per_channel(x2)
    assert set(np.nonzero(q0 != q1)[1]) == {11} and set(np.nonzero(s0 != s1)[0]) == {11}


def pin_swiglu(o):
    """silu(g) - silu(-g) = g (sigmoid(g) + sigmoid(-g) = 1), silu(ln 3) =
    0.75 ln 3, silu(0) = 0; h rounds silu(gate) * up to BF16 with the gate in
    the first half of each row and the up projection in the second; the
    codes are the 1x128 quantisation of h."""
    g = np.linspace(-20, 20, 4001)
    d = o.silu_mul(g, np.ones_like(g)) - o.silu_mul(-g, np.ones_like(g))
    assert np.all(np.abs(d - g) <= 1e-14 * np.maximum(1, np.abs(g)))
    assert abs(o.silu_mul(np.log(3.0), 1.0) - 0.75 * np.log(3.0)) < 1e-15 and o.silu_mul(0.0, 5.0) == 0.0
    rng = np.random.default_rng(71)
    gate = (rng.standard_normal((3, 256)) * 2).astype(np.float32)
    up = rng.standard_normal((3, 256)).astype(np.float32)
    h, qa, sa = o.swiglu_quant_act_1x128(np.concatenate([gate, up], axis=1))
    want = gate.astype(np.float64) / (1 + np.exp(-gate.astype(np.float64))) * up
    assert np.array_equal(h, o.bf16_round(want.astype(np.float32)))
    q2, s2 = o.quant_act_1x128(h)
    assert np.array_equal(qa, q2) and np.array_equal(sa, s2)
    h0, _, _ = o.swiglu_quant_act_1x128(np.concatenate([np.zeros_like(gate), up], axis=1))
    assert np.all(h0 == 0)


def pin_gemm_residual(o):
    """Residual epilogue: all-zero weights give back the residual exactly
    (every weight group has s = 0 and codes 0); constant operands give the
    closed form K (448 s_x)(448 s_w) plus the residual."""
    rng = np.random.default_rng(43)
    M, N, K = 6, 256, 256
    x = rng.standard_normal((M, K)).astype(np.float32)
    r = o.bf16_round((rng.standard_normal((M, N)) * 3.0).astype(np.float32))
    qa, sa = o.quant_act_1x128(x)
    qz, sz = o.quant_weight_128x128(np.zeros((N, K), dtype=np.float32))
    assert np.array_equal(o.blockscaled_gemm_residual(qa, sa, qz, sz, r), r.astype(np.float64))
    xc = np.full((M, K), np.float32(2.0), dtype=np.float32)
    wc = np.full((N, K), np.float32(-0.25), dtype=np.float32)
    qa, sa = o.quant_act_1x128(xc)
    qw, sw = o.quant_weight_128x128(wc)
    want = -(K * (448.0 * float(sa[0, 0])) * (448.0 * float(sw[0, 0]))) + r.astype(np.float64)
    assert np.array_equal(o.blockscaled_gemm_residual(qa, sa, qw, sw, r), want)


def pin_act_dequant(o):
    """dequant of the cached 1x128 activation: quant then dequant stays within
    half an E4M3 ulp of each group (times its scale) plus the BF16 rounding;
    with scales constant over 128x128 blocks it equals the weight dequant
    (which indexes its scales the other way round); the float32 product is
    rounded to BF16 once more (0x39 = 1.125 times 1.0078125 -> 1.1328125)."""
    rng = np.random.default_rng(71)
    x = (rng.standard_normal((256, 384)) * np.exp(rng.standard_normal((256, 1)) * 3)).astype(np.float32)
    x[5, 128:256] = 0.0
    qa, sa = o.quant_act_1x128(x)
    y = o.dequant_act_1x128_bf16(qa, sa).astype(np.float64)
    s = np.repeat(sa.T.astype(np.float64), 128, axis=1)
    v = np.abs(x.astype(np.float64)) / np.where(s > 0, s, 1)
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
    ulp = np.where(v < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))
    bound = 0.5 * ulp * s * (1 + 2.0 ** -20) + np.abs(x) * 2.0 ** -8 + 1e-300
    assert np.all(np.abs(y - x) <= bound)
    assert np.all(y[5, 128:256] == 0.0)
    q = rng.integers(0, 256, (256, 384)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x11  # no NaN codes
    sw = rng.uniform(0.5, 2.0, (2, 3)).astype(np.float32)
    sa_blocks = np.repeat(sw.T, 128, axis=1)  # sa[kb, m] = sw[m // 128, kb]
    assert np.array_equal(o.dequant_act_1x128_bf16(q, sa_blocks).view(np.uint32),
                          o.dequant_weight_128x128_bf16(q, sw).view(np.uint32))
    q1 = np.full((3, 128), 0x39, dtype=np.uint8)
    got = o.dequant_act_1x128_bf16(q1, np.full((1, 4), 1.0078125, dtype=np.float32))
    assert got.shape == (3, 128) and np.all(got == np.float32(1.1328125))


def pin_requant_transpose_identity(o):
    """When every scale is a power of two, constant over each 128x128 tile,
    and each column of each tile holds a +-448 code, the dequantised values
    are exact and every (128-token, channel) group has amax 448 s: the
    requantised codes of X^T are the cached codes transposed, bit for bit,
    and its scales are the tile scales in the [M/128, K] layout."""
    rng = np.random.default_rng(73)
    M, K = 256, 384
    q = rng.integers(0, 256, (M, K)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x22
    q[rng.integers(0, 128, K), np.arange(K)] = 0x7E            # a +448 code in every column of tile row 0
    q[128 + rng.integers(0, 128, K), np.arange(K)] = 0xFE      # a -448 code in every column of tile row 1
    e = rng.integers(-12, 12, (K // 128, M // 128))            # exponent of tile (kb, mb)
    sa = np.repeat(np.ldexp(1.0, e), 128, axis=1).astype(np.float32)  # [K/128, M]
    qt, st = o.requant_act_1x128_t(q, sa)
    assert qt.shape == (K, M) and st.shape == (M // 128, K)
    assert np.array_equal(qt, q.T)
    assert np.array_equal(st, np.repeat(np.ldexp(1.0, e.T), 128, axis=1).astype(np.float32))


def pin_backward_cached(o):
    """With X exactly representable by its 1x128 quantisation (each group a
    power of two times E4M3 values, one of them +-448), the cached-activation
    backward equals the BF16-activation backward exactly; on general X its dW
    stays within the E4M3 worst case of the unquantised product."""
    rng = np.random.default_rng(79)
    M, N, K = 256, 128, 256
    codes = rng.integers(0, 256, (M, K)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x30
    codes[np.arange(M), rng.integers(0, 128, M)] = 0x7E
    codes[np.arange(M), 128 + rng.integers(0, 128, M)] = 0xFE
    e = rng.integers(-6, 6, (M, K // 128))
    x = (o.e4m3_decode(codes) * np.repeat(np.ldexp(1.0, e), 128, axis=1)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    dy = rng.standard_normal((M, N)).astype(np.float32)
    qa, sa = o.quant_act_1x128(x)
    assert np.array_equal(qa, codes)
    dx_c, dw_c = o.linear_backward_cached(qa, sa, w, dy)
    dx, dw = o.linear_backward(x, w, dy)
    assert np.array_equal(dx_c, dx) and np.array_equal(dw_c, dw)
    xg = rng.standard_normal((M, K)).astype(np.float32)
    qg, sg = o.quant_act_1x128(xg)
    _, dw_g = o.linear_backward_cached(qg, sg, w, dy)
    exact = dy.astype(np.float64).T @ xg.astype(np.float64)
    # X goes through two E4M3 roundings (1x128, then 128 tokens), dY through one
    mag = np.abs(dy.astype(np.float64)).T @ np.abs(xg.astype(np.float64))
    rel = (1 + 2.0 ** -4) ** 2 * (1 + 2.0 ** -8) * (1 + 2.0 ** -4) - 1
    assert np.all(np.abs(dw_g - exact) <= rel * mag + 2.0 ** -6)


ALL_PINS = [
    pin_dequant_float64,
    pin_act_dequant,
    pin_requant_transpose_identity,
    pin_backward_cached,
    pin_gemm_residual,
    pin_codec_format_points,
    pin_codec_roundtrip,
    pin_codec_ties,
    pin_codec_saturation,
    pin_codec_sign_of_zero,
    pin_codec_vs_torch,
    pin_fl32_div_exact,
    pin_scale_definition,
    pin_quant_worked_example,
    pin_quant_exact_ties,
    pin_amax_maps_to_448,
    pin_quant_error_bound,
    pin_quant_pow2_invariance,
    pin_quant_locality,
    pin_weight_structure,
    pin_gemm_bruteforce,
    pin_gemm_closed_form,
    pin_gemm_onehot,
    pin_gemm_linearity,
    pin_gemm_rows_columns,
    pin_grouped,
    pin_bf16_round,
    pin_dequant_roundtrip,
    pin_rowscaled_bruteforce,
    pin_rowscaled_reduces_to_blockscaled,
    pin_transposed_quant_structure,
    pin_backward_error_bound,
    pin_backward_linearity,
    pin_e5m6_format,
    pin_e5m6_roundtrip_and_ties,
    pin_per_token_and_channel,
    pin_swiglu,
]
