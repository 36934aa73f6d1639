"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Every mutant is a one-line textual change to the oracle source, executed as
a throw-away module on the CPU; the real oracle is never modified.  This
shows the pins in oracle_pins.py are strong enough to catch a dropped term,
a wrong sign, index or rounding rule, or a transposed operand.
"""
import os
import types

import pytest

from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "fp8_oracle.py")

MUTANTS = {
    "ties_away_from_zero": (
        "take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))",
        "take_hi = (d_hi < d_lo) | (d_hi == d_lo)"),
    "ties_toward_zero": (
        "take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))",
        "take_hi = (d_hi < d_lo)"),
    "no_saturation": (
        "code = np.where(saturate, 0x7E, code)",
        "code = np.where(saturate, 0x7F, code)"),
    "sign_of_zero_dropped": (
        "code = code | (np.signbit(v).astype(np.int64) << 7)",
        "code = code | ((v < 0).astype(np.int64) << 7)"),
    "scale_by_reciprocal": (
        "s = fl32_div(amax, np.float32(E4M3_MAX))",
        "s = (amax * np.float32(1.0 / 448.0)).astype(np.float32)"),
    "quantise_by_multiply": (
        "v = fl32_div(g, s[..., None])",
        "v = (g * fl32_div(np.float32(1.0), s)[..., None]).astype(np.float32)"),
    "zero_group_not_cleared": (
        "codes[s == 0] = 0",
        "pass"),
    "amax_without_abs": (
        "amax = np.max(np.abs(g), axis=-1)",
        "amax = np.max(g, axis=-1)"),
    "decode_bias_8": (
        "normal = np.ldexp(1.0 + man / 8.0, exp - 7)",
        "normal = np.ldexp(1.0 + man / 8.0, exp - 8)"),
    "decode_subnormal_exponent": (
        "subnormal = np.ldexp(man / 8.0, -6)",
        "subnormal = np.ldexp(man / 8.0, -7)"),
    "weight_blocks_not_transposed": (
        "blocks = w.reshape(NB, GROUP, KB, GROUP).transpose(0, 2, 1, 3).reshape(NB, KB, GROUP * GROUP)",
        "blocks = w.reshape(NB, KB, GROUP * GROUP)"),
    "act_scales_not_transposed": (
        "return codes.reshape(M, K), np.ascontiguousarray(s.T)",
        "return codes.reshape(M, K), np.ascontiguousarray(s.T[::-1])"),
    "weight_scale_of_chunk_0": (
        "col_scale = np.repeat(sw[:, kb].astype(np.float64), GROUP)",
        "col_scale = np.repeat(sw[:, 0].astype(np.float64), GROUP)"),
    "act_scale_of_chunk_0": (
        "row_scale = sa[kb, :M].astype(np.float64)",
        "row_scale = sa[0, :M].astype(np.float64)"),
    "act_scale_dropped": (
        "y += chunk * (row_scale[:, None] * col_scale[None, :])",
        "y += chunk * (col_scale[None, :] + 0 * row_scale[:, None])"),
    "weight_scale_rows_swapped": (
        "col_scale = np.repeat(sw[:, kb].astype(np.float64), GROUP)",
        "col_scale = np.repeat(sw[::-1, kb].astype(np.float64), GROUP)"),
    "operand_columns_reversed": (
        "chunk = a @ b.T",
        "chunk = (a @ b.T)[:, ::-1]"),
    "negated_product": (
        "chunk = a @ b.T",
        "chunk = -(a @ b.T)"),
    "bf16_round_truncates": (
        "r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16",
        "r = u >> 16"),
    "bf16_round_ties_away": (
        "r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16",
        "r = (u + 0x8000) >> 16"),
    "dequant_scale_of_first_block": (
        "scale = np.repeat(np.repeat(np.asarray(sw, dtype=np.float32), GROUP, axis=0), GROUP, axis=1)",
        "scale = np.full(qw.shape, np.asarray(sw, dtype=np.float32).flat[0], dtype=np.float32)"),
    "dequant64_scale_rows_reversed": (
        "scale = np.repeat(np.repeat(np.asarray(sw, dtype=np.float64), GROUP, axis=0), GROUP, axis=1)",
        "scale = np.repeat(np.repeat(np.asarray(sw, dtype=np.float64)[::-1], GROUP, axis=0), GROUP, axis=1)"),
    "dequant64_scale_of_first_block": (
        "scale = np.repeat(np.repeat(np.asarray(sw, dtype=np.float64), GROUP, axis=0), GROUP, axis=1)",
        "scale = np.full((N, K), np.asarray(sw, dtype=np.float64).flat[0])"),
    "dequant64_scale_dropped": (
        "return e4m3_decode(qw) * scale",
        "return e4m3_decode(qw) + 0 * scale"),
    "rowscaled_column_scale_of_chunk_0": (
        "y += chunk * (sa[kb, :M].astype(np.float64)[:, None] * sb[kb, :N].astype(np.float64)[None, :])",
        "y += chunk * (sa[kb, :M].astype(np.float64)[:, None] * sb[0, :N].astype(np.float64)[None, :])"),
    "rowscaled_column_scale_dropped": (
        "y += chunk * (sa[kb, :M].astype(np.float64)[:, None] * sb[kb, :N].astype(np.float64)[None, :])",
        "y += chunk * (sa[kb, :M].astype(np.float64)[:, None] + 0 * sb[kb, :N].astype(np.float64)[None, :])"),
    "backward_weight_not_transposed": (
        "dx = blockscaled_gemm(qdy, sdy, qwt, swt)",
        "dx = blockscaled_gemm(qdy, sdy, qw, sw)"),
    "backward_wgrad_operands_swapped": (
        "dw = blockscaled_gemm_rowscaled(qdyt, sdyt, qxt, sxt)",
        "dw = blockscaled_gemm_rowscaled(qdyt, sdyt, qdyt, sdyt)"),
    "transposed_quant_not_transposed": (
        "return quant_act_1x128(np.ascontiguousarray(x.T))",
        "return quant_act_1x128(x)"),
    "e5m6_bias_16": (
        "normal = np.ldexp(1.0 + man / 64.0, exp - 15)",
        "normal = np.ldexp(1.0 + man / 64.0, exp - 16)"),
    "e5m6_ties_away": (
        "take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_E5M6_POS_CODES[hi] % 2 == 0))",
        "take_hi = (d_hi <= d_lo)"),
    "per_channel_is_per_token": (
        "codes, s = _quantise_groups(np.ascontiguousarray(x.T))\n    return np.ascontiguousarray(codes.T), s",
        "codes, s = _quantise_groups(x)\n    return codes, s"),
    "swiglu_gate_up_swapped": (
        "h = bf16_round(silu_mul(gu[:, :F], gu[:, F:]).astype(np.float32))",
        "h = bf16_round(silu_mul(gu[:, F:], gu[:, :F]).astype(np.float32))"),
    "silu_sign_flipped": (
        "return g / (1.0 + np.exp(-g)) * u",
        "return g / (1.0 + np.exp(g)) * u"),
    "residual_subtracted": (
        "return blockscaled_gemm(qa, sa, qw, sw) + np.asarray(r, dtype=np.float64)",
        "return blockscaled_gemm(qa, sa, qw, sw) - np.asarray(r, dtype=np.float64)"),
    "residual_dropped": (
        "return blockscaled_gemm(qa, sa, qw, sw) + np.asarray(r, dtype=np.float64)",
        "return blockscaled_gemm(qa, sa, qw, sw)"),
    "act_dequant_scale_rows_reversed": (
        "scale = np.repeat(np.ascontiguousarray(sa.T), GROUP, axis=1)",
        "scale = np.repeat(np.ascontiguousarray(sa.T[::-1]), GROUP, axis=1)"),
    "act_dequant_not_rounded_to_bf16": (
        "x = bf16_round(prod)",
        "x = prod"),
    "requant_not_transposed": (
        "return quant_act_1x128_t(dequant_act_1x128_bf16(qa, sa))",
        "return quant_act_1x128(dequant_act_1x128_bf16(qa, sa))"),
    "cached_backward_requantises_dy": (
        "return _linear_backward_from(requant_act_1x128_t(qa, sa), w, dy)",
        "return _linear_backward_from(quant_act_1x128_t(dy), w, dy)"),
    "grouped_wrong_weight_scales": (
        "y[r0:r1] = blockscaled_gemm(qa[r0:r1], sa[:, r0:r1], qw[g], sw[g])",
        "y[r0:r1] = blockscaled_gemm(qa[r0:r1], sa[:, r0:r1], qw[g], sw[0])"),
    "grouped_wrong_rows_for_scales": (
        "y[r0:r1] = blockscaled_gemm(qa[r0:r1], sa[:, r0:r1], qw[g], sw[g])",
        "y[r0:r1] = blockscaled_gemm(qa[r0:r1], sa[:, :r1 - r0], qw[g], sw[g])"),
}


def _mutant_module(old, new):
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site not found exactly once: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = SRC
    exec(compile(src.replace(old, new), SRC + " (mutant)", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    mod = _mutant_module(old, new)
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception:
            return  # caught
    pytest.fail(f"mutant {name} passed every pin")
