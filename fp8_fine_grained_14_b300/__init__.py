"""Fine-grained FP8 block-scaled linear layer for B300 (sm_103a).

The compute path is the C-ABI library libfp8bs.so (include/fp8bs.h); the
names below are its thin ctypes binding, loaded on first use.  `workloads`
(seeded synthetic inputs) needs no GPU and no library.
"""
import importlib

from . import workloads  # noqa: F401

_API = (
    "fp8_quant_act_1x128",
    "fp8_quant_weight_128x128",
    "fp8_blockscaled_gemm",
    "fp8_blockscaled_gemm_noalloc",
    "fp8_blockscaled_gemm_workspace_bytes",
    "fp8_blockscaled_gemm_residual",
    "fp8_blockscaled_grouped_gemm",
    "fp8_dequant_weight_128x128",
    "fp8_quant_act_1x128_t",
    "fp8_requant_act_1x128_t",
    "fp8_pack_weight_128x128",
    "fp8_blockscaled_gemm_packed",
    "fp8_transpose_weight_128x128",
    "fp8_blockscaled_gemm_rowscaled",
    "linear_backward",
    "fp8_quant_per_token",
    "fp8_quant_per_channel",
    "e5m6_encode",
    "e5m6_decode",
    "fp8_swiglu_quant_act_1x128",
    "fp8bs_last_device_error",
    "fp8bs_set_wait_timeout_ns",
    "fp8bs_selftest_wait_timeout",
    "fp8bs_stream_timestamp",
    "linear_forward",
    "HostPipeline",
    "ld_sa_for",
    "Fp8bsError",
)


def __getattr__(name):
    if name in _API or name == "binding":
        binding = importlib.import_module(__name__ + ".binding")
        return binding if name == "binding" else getattr(binding, name)
    raise AttributeError(name)
