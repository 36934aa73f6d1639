"""The C-ABI library on a CPU-only host: it loads, exports every function
include/fp8bs.h declares, and rejects bad arguments synchronously, before
any CUDA call (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:fp8|fp8bs)_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from fp8_fine_grained_14_b300 import binding

    return binding.lib


def test_header_declares_the_four_entry_points():
    names = _declared_functions()
    for n in ("fp8_quant_act_1x128", "fp8_quant_weight_128x128", "fp8_blockscaled_gemm",
              "fp8_blockscaled_grouped_gemm"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_export():
    from fp8_fine_grained_14_b300 import binding

    assert set(_declared_functions()) <= set(binding.EXPORTS)


def test_header_preamble_discloses_owned_memory():
    """The conventions every caller reads first name all memory the library
    owns: the status word, the no-alloc GEMM's static array and the
    split-K workspace pool, with its bound and stream rule."""
    text = open(HEADER).read()
    preamble = text[:text.index("#ifndef FP8BS_H")]
    for phrase in ("status word", "static scratch array", "memory pool", "128 KiB per SM", "on its stream",
                   "fp8_blockscaled_gemm_workspace_bytes"):
        assert phrase in preamble, phrase
    gemm_doc = text[:text.index("fp8bs_status fp8_blockscaled_gemm(")]
    gemm_doc = gemm_doc[gemm_doc.rindex("/*"):]
    assert "pool" in gemm_doc and "workspace" in gemm_doc


@pytest.mark.parametrize("args,expect", [
    ((128, 256, 256, None), 1),        # null out
    ((-1, 256, 256, "out"), 1),        # negative M
    ((128, 100, 256, "out"), 3),       # N % 128
    ((128, 256, 0, "out"), 3),         # K == 0
    ((0, 256, 256, "out"), 0),         # M == 0: nothing to split, no device query
])
def test_workspace_query_validation(lib, args, expect):
    out = ctypes.c_size_t(12345)
    M, N, K, o = args
    st = lib.fp8_blockscaled_gemm_workspace_bytes(M, N, K, ctypes.byref(out) if o else None)
    assert st == expect
    if o and expect in (0, 3):
        assert out.value == 0


def test_status_strings(lib):
    for code in range(6):
        assert lib.fp8bs_status_string(code)
    assert lib.fp8bs_status_string(99) == b"unknown status"


P = ctypes.c_void_p
A16 = P(0x10000)  # aligned dummy address; validation fails before any use


@pytest.mark.parametrize("args,expect", [
    ((A16, 4, 100, 100, A16, 112, A16, 4, None), 3),     # K % 128
    ((A16, 4, 0, 0, A16, 0, A16, 4, None), 3),           # K == 0
    ((A16, -1, 128, 128, A16, 128, A16, 4, None), 1),    # negative M
    ((A16, 4, 128, 64, A16, 128, A16, 4, None), 1),      # ldx < K
    ((A16, 8, 128, 128, A16, 128, A16, 4, None), 1),     # ld_sa < M
    ((A16, 0, 128, 128, None, 128, None, 0, None), 0),   # M == 0 is a no-op
    ((None, 4, 128, 128, A16, 128, A16, 4, None), 1),    # null x
    ((P(0x10002), 4, 128, 128, A16, 128, A16, 4, None), 2),  # misaligned x
    ((A16, 4, 128, 132, A16, 144, A16, 4, None), 2),     # ldx % 8
    ((A16, 4, 128, 128, A16, 136, A16, 4, None), 2),     # ldq % 16
    ((A16, 3, 128, 128, A16, 128, A16, 6, None), 2),     # ld_sa % 4
])
def test_quant_act_validation(lib, args, expect):
    assert lib.fp8_quant_act_1x128(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((A16, 100, 128, 128, A16, 128, A16, None), 3),      # N % 128
    ((A16, 128, 100, 128, A16, 128, A16, None), 3),      # K % 128
    ((A16, 0, 128, 128, A16, 128, A16, None), 3),        # N == 0
    ((A16, 128, 128, 128, None, 128, A16, None), 1),
    ((A16, 128, 128, 128, A16, 128, P(0x10004), None), 2),
])
def test_quant_weight_validation(lib, args, expect):
    assert lib.fp8_quant_weight_128x128(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((A16, 128, A16, 4, A16, 128, A16, A16, 128, 1, 100, 128, None), 3),   # N % 128
    ((A16, 128, A16, 4, A16, 128, A16, A16, 128, 1, 128, 64, None), 3),    # K % 128
    ((A16, 128, A16, 4, A16, 128, A16, A16, 128, 0, 128, 128, None), 0),   # M == 0
    ((A16, 128, A16, 4, A16, 128, A16, A16, 64, 1, 128, 128, None), 1),    # ldy < N
    ((A16, 128, A16, 4, A16, 128, A16, P(0x10008), 128, 1, 128, 128, None), 2),
    ((A16, 128, A16, 4, A16, 136, A16, A16, 128, 1, 128, 128, None), 2),   # ldqw % 16
    ((None, 128, A16, 4, A16, 128, A16, A16, 128, 1, 128, 128, None), 1),
])
def test_gemm_validation(lib, args, expect):
    assert lib.fp8_blockscaled_gemm(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((A16, 128, 100, 128, A16, A16, 128, None), 3),      # K % 128
    ((A16, 0, 128, 128, A16, A16, 128, None), 3),        # N == 0
    ((A16, 128, 128, 64, A16, A16, 128, None), 1),       # ldq < K
    ((A16, 128, 128, 128, A16, A16, 64, None), 1),       # ldy < K
    ((None, 128, 128, 128, A16, A16, 128, None), 1),     # null codes
    ((A16, 128, 128, 136, A16, A16, 128, None), 2),      # ldq % 16
    ((A16, 128, 128, 128, A16, P(0x10008), 128, None), 2),  # misaligned y
    ((A16, 128, 128, 128, P(0x10002), A16, 128, None), 2),  # misaligned scales
])
def test_dequant_validation(lib, args, expect):
    assert lib.fp8_dequant_weight_128x128(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((0, A16, 10, A16, 128, A16, 12, A16, A16, A16, 128, 128, 128, None), 1),      # G == 0
    ((2, None, 10, A16, 128, A16, 12, A16, A16, A16, 128, 128, 128, None), 1),     # null offsets
    ((2, A16, 10, A16, 128, A16, 12, A16, A16, A16, 128, 100, 128, None), 3),      # N % 128
    ((2, A16, 0, A16, 128, A16, 0, A16, A16, A16, 128, 128, 128, None), 0),        # M_total == 0
    ((2, P(0x10002), 10, A16, 128, A16, 12, A16, A16, A16, 128, 128, 128, None), 2),
    ((2, A16, 10, A16, 128, A16, 8, A16, A16, A16, 128, 128, 128, None), 1),       # ld_sa < M_total
])
def test_grouped_validation(lib, args, expect):
    assert lib.fp8_blockscaled_grouped_gemm(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((A16, 128, A16, 4, A16, 128, A16, None, 128, A16, 128, 1, 128, 128, None), 1),        # null residual
    ((A16, 128, A16, 4, A16, 128, A16, A16, 120, A16, 128, 1, 128, 128, None), 1),         # ldr < N
    ((A16, 128, A16, 4, A16, 128, A16, A16, 128, A16, 136, 1, 128, 128, None), 1),         # in place, ldr != ldy
    ((A16, 128, A16, 4, A16, 128, A16, P(0x10002), 128, A16, 128, 1, 128, 128, None), 2),  # misaligned residual
    ((A16, 128, A16, 4, A16, 128, A16, P(0x20000), 132, A16, 128, 1, 128, 128, None), 2),  # ldr % 8
    ((A16, 128, A16, 4, A16, 128, A16, P(0x20000), 128, A16, 128, 1, 100, 128, None), 3),  # N % 128
    ((A16, 128, A16, 4, A16, 128, A16, None, 0, A16, 128, 0, 128, 128, None), 0),          # M == 0
])
def test_gemm_residual_validation(lib, args, expect):
    assert lib.fp8_blockscaled_gemm_residual(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((A16, 128, A16, 128, 100, 128, A16, 128, A16, 128, None), 3),        # M % 128
    ((A16, 128, A16, 128, 128, 100, A16, 128, A16, 128, None), 3),        # K % 128
    ((A16, 128, A16, 64, 128, 128, A16, 128, A16, 128, None), 1),         # ld_sa < M
    ((A16, 64, A16, 128, 128, 128, A16, 128, A16, 128, None), 1),         # ldqa < K
    ((None, 128, A16, 128, 128, 128, A16, 128, A16, 128, None), 1),       # null codes
    ((A16, 128, P(0x10004), 128, 128, 128, A16, 128, A16, 128, None), 2),  # scales not 16-byte aligned
    ((A16, 136, A16, 128, 128, 128, A16, 128, A16, 128, None), 2),        # ldqa % 16
    ((A16, 128, A16, 130, 128, 128, A16, 128, A16, 128, None), 2),        # ld_sa % 4
    ((A16, 128, A16, 0, 0, 128, A16, 0, A16, 128, None), 0),              # M == 0
])
def test_requant_validation(lib, args, expect):
    assert lib.fp8_requant_act_1x128_t(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((A16, 100, 128, 128, A16, None), 3),          # N % 128
    ((A16, 128, 100, 128, A16, None), 3),          # K % 128
    ((A16, 128, 128, 64, A16, None), 1),           # ldq < K
    ((None, 128, 128, 128, A16, None), 1),         # null codes
    ((A16, 128, 128, 128, P(0x10008), None), 2),   # misaligned output
    ((A16, 128, 128, 136, A16, None), 2),          # ldq % 16
])
def test_pack_validation(lib, args, expect):
    assert lib.fp8_pack_weight_128x128(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((A16, 128, A16, 4, A16, A16, A16, 128, 1, 100, 128, None), 3),       # N % 128
    ((A16, 128, A16, 4, A16, A16, A16, 128, 0, 128, 128, None), 0),       # M == 0
    ((A16, 128, A16, 4, None, A16, A16, 128, 1, 128, 128, None), 1),     # null packed weights
    ((A16, 128, A16, 4, P(0x10008), A16, A16, 128, 1, 128, 128, None), 2),  # misaligned packed weights
    ((A16, 128, A16, 4, A16, A16, A16, 120, 1, 128, 128, None), 1),       # ldy < N
])
def test_gemm_packed_validation(lib, args, expect):
    assert lib.fp8_blockscaled_gemm_packed(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((None, 0, None), 1),        # null destination
    ((P(0x10004), 1, None), 2),  # not 8-byte aligned
])
def test_stream_timestamp_validation(lib, args, expect):
    assert lib.fp8bs_stream_timestamp(*args) == expect


def test_header_is_plain_c(tmp_path):
    """include/fp8bs.h compiles as C (no C++ in the ABI)."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    src = tmp_path / "use_header.c"
    src.write_text('#include "fp8bs.h"\nint main(void) { return fp8bs_status_string(FP8BS_OK) == 0; }\n')
    res = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
                          "-I", cuda_inc, str(src)], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
