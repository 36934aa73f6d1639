"""CPU oracle of the fine-grained FP8 block-scaled linear layer.

Test infrastructure only: imported by the tests, the smoke check and the
benchmark's CPU baseline leg, never by the product path.
"""
from .fp8_oracle import (  # noqa: F401
    E4M3_MAX,
    E5M6_MAX,
    GROUP,
    blockscaled_gemm,
    blockscaled_gemm_residual,
    blockscaled_gemm_rowscaled,
    blockscaled_grouped_gemm,
    bf16_round,
    dequant_act_1x128_bf16,
    dequant_weight_128x128,
    dequant_weight_128x128_bf16,
    e4m3_decode,
    e4m3_encode_rne_satfinite,
    e5m6_decode,
    e5m6_encode_rne_satfinite,
    fl32_div,
    linear_backward,
    linear_backward_cached,
    linear_forward,
    quant_act_1x128,
    quant_act_1x128_t,
    quant_per_channel,
    quant_per_token,
    silu_mul,
    swiglu_quant_act_1x128,
    quant_weight_128x128,
    requant_act_1x128_t,
    transpose_weight_128x128,
)
