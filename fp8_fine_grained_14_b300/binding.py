"""ctypes binding of libfp8bs.so (declared in include/fp8bs.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (torch provides device memory
and the current stream); outputs are allocated here when not supplied.
There is no CPU fallback: importing this module fails loudly when the
library has not been built, and every call fails on a host without a GPU.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8bs.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m fp8_fine_grained_14_b300.build` "
        "(or __graft_entry__.build()); there is no fallback implementation")

lib = ctypes.CDLL(LIB_PATH)

_i64, _i32, _u64, _p = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_void_p

STATUS = {0: "FP8BS_OK", 1: "FP8BS_ERR_INVALID_ARG", 2: "FP8BS_ERR_MISALIGNED",
          3: "FP8BS_ERR_UNSUPPORTED_SHAPE", 4: "FP8BS_ERR_CUDA", 5: "FP8BS_ERR_TIMEOUT"}
EXPORTS = {
    "fp8_quant_act_1x128": [_p, _i64, _i64, _i64, _p, _i64, _p, _i64, _p],
    "fp8_quant_weight_128x128": [_p, _i64, _i64, _i64, _p, _i64, _p, _p],
    "fp8_blockscaled_gemm": [_p, _i64, _p, _i64, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _p],
    "fp8_blockscaled_gemm_noalloc": [_p, _i64, _p, _i64, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _p],
    "fp8_blockscaled_gemm_residual": [_p, _i64, _p, _i64, _p, _i64, _p, _p, _i64, _p, _i64, _i64, _i64, _i64, _p],
    "fp8_blockscaled_grouped_gemm": [_i32, _p, _i64, _p, _i64, _p, _i64, _p, _p, _p, _i64, _i64, _i64, _p],
    "fp8_blockscaled_gemm_f32": [_p, _i64, _p, _i64, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _p],
    "fp8_blockscaled_grouped_gemm_f32": [_i32, _p, _i64, _p, _i64, _p, _i64, _p, _p, _p, _i64, _i64, _i64, _p],
    "fp8_dequant_weight_128x128": [_p, _i64, _i64, _i64, _p, _p, _i64, _p],
    "fp8_quant_act_1x128_t": [_p, _i64, _i64, _i64, _p, _i64, _p, _i64, _p],
    "fp8_requant_act_1x128_t": [_p, _i64, _p, _i64, _i64, _i64, _p, _i64, _p, _i64, _p],
    "fp8_pack_weight_128x128": [_p, _i64, _i64, _i64, _p, _p],
    "fp8_blockscaled_gemm_packed": [_p, _i64, _p, _i64, _p, _p, _p, _i64, _i64, _i64, _i64, _p],
    "fp8_quant_per_token": [_p, _i64, _i64, _i64, _p, _i64, _p, _p],
    "fp8_quant_per_channel": [_p, _i64, _i64, _i64, _p, _i64, _p, _p],
    "fp8bs_e5m6_encode_bf16": [_p, _i64, _p, _p],
    "fp8bs_e5m6_decode_bf16": [_p, _i64, _p, _p],
    "fp8_swiglu_quant_act_1x128": [_p, _i64, _i64, _i64, _p, _i64, _p, _i64, _p, _i64, _p],
    "fp8_transpose_weight_128x128": [_p, _i64, _i64, _i64, _p, _p, _i64, _p, _p],
    "fp8_blockscaled_gemm_rowscaled": [_p, _i64, _p, _i64, _p, _i64, _p, _i64, _p, _i64, _i64, _i64, _i64, _p],
    "fp8_blockscaled_gemm_rowscaled_f32": [_p, _i64, _p, _i64, _p, _i64, _p, _i64, _p, _i64, _i64, _i64, _i64,
                                           _p],
    "fp8_blockscaled_gemm_workspace_bytes": [_i64, _i64, _i64, ctypes.POINTER(ctypes.c_size_t)],
    "fp8bs_status_string": [ctypes.c_int],
    "fp8bs_last_error_detail": [],
    "fp8bs_last_device_error": [_p],
    "fp8bs_set_wait_timeout_ns": [_u64],
    "fp8bs_selftest_wait_timeout": [_u64, _p],
    "fp8bs_stream_timestamp": [_p, ctypes.c_int, _p],
}
for _name, _args in EXPORTS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = ctypes.c_int
lib.fp8bs_status_string.restype = ctypes.c_char_p
lib.fp8bs_last_error_detail.restype = ctypes.c_char_p
lib.fp8bs_set_wait_timeout_ns.restype = None


class Fp8bsError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = lib.fp8bs_status_string(status).decode()
        detail = lib.fp8bs_last_error_detail().decode() if status == 4 else ""
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({msg}){': ' + detail if detail else ''}")


def _check(fn, status):
    if status != 0:
        raise Fp8bsError(fn, status)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else ctypes.c_void_p(0)


def _require(t, dtype, name, ndim):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.dim() != ndim or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA {dtype} tensor with {ndim} dims")
    if t.stride(-1) != 1:
        raise ValueError(f"{name} must have unit stride along its last dimension")


def _require_min(t, dtype, name, rows, cols):
    """A 2-D buffer the library reads or writes through its row stride: it
    must hold at least `rows` rows of `cols` elements, since the C ABI sees
    only the pointer and the stride."""
    _require(t, dtype, name, 2)
    if t.shape[0] < rows or t.shape[1] < cols:
        raise ValueError(f"{name} must be at least [{rows}, {cols}], got {list(t.shape)}")


def _require_count(t, name, count, dtype=torch.float32):
    """A contiguous buffer the library indexes densely (block scales, per-row
    or per-column scales): at least `count` elements."""
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA {dtype} tensor")
    if t.numel() < count:
        raise ValueError(f"{name} must hold at least {count} elements, got {t.numel()}")


def ld_sa_for(m: int) -> int:
    """Row stride of the transposed activation-scale matrix: M rounded up to 4."""
    return (m + 3) // 4 * 4


def fp8_quant_act_1x128(x, qa=None, sa=None, stream=None):
    """x bf16 [M, K] -> (qa uint8 [M, K] E4M3 codes, sa float32 [K/128, ld_sa]).

    sa[kb, m] is the scale of row m, channels 128*kb..; ld_sa = M rounded up
    to a multiple of 4 unless `sa` is supplied."""
    _require(x, torch.bfloat16, "x", 2)
    M, K = x.shape
    if qa is None:
        qa = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sa is None:
        sa = torch.empty((K // 128, ld_sa_for(M)), dtype=torch.float32, device=x.device)
    _require_min(qa, torch.uint8, "qa", M, K)
    _require_min(sa, torch.float32, "sa", K // 128, M)
    st = lib.fp8_quant_act_1x128(_ptr(x), M, K, x.stride(0), _ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0),
                                 _stream(stream))
    _check("fp8_quant_act_1x128", st)
    return qa, sa


def fp8_quant_weight_128x128(w, qw=None, sw=None, stream=None):
    """w bf16 [N, K] -> (qw uint8 [N, K], sw float32 [N/128, K/128]).
    A stack of experts [G, N, K] is accepted and quantised as [G*N, K]."""
    if isinstance(w, torch.Tensor) and w.dim() == 3:
        G, N, K = w.shape
        qw3 = qw if qw is not None else torch.empty((G, N, K), dtype=torch.uint8, device=w.device)
        sw3 = sw if sw is not None else torch.empty((G, N // 128, K // 128), dtype=torch.float32, device=w.device)
        fp8_quant_weight_128x128(w.reshape(G * N, K), qw3.view(G * N, K), sw3.view(G * N // 128, K // 128),
                                 stream=stream)
        return qw3, sw3
    _require(w, torch.bfloat16, "w", 2)
    N, K = w.shape
    if qw is None:
        qw = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    if sw is None:
        sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    _require_min(qw, torch.uint8, "qw", N, K)
    _require_count(sw, "sw", (N // 128) * (K // 128))
    st = lib.fp8_quant_weight_128x128(_ptr(w), N, K, w.stride(0), _ptr(qw), qw.stride(0), _ptr(sw),
                                      _stream(stream))
    _check("fp8_quant_weight_128x128", st)
    return qw, sw


def fp8_blockscaled_gemm(qa, sa, qw, sw, y=None, stream=None, out_dtype=torch.bfloat16):
    """Block-scaled FP8 GEMM: Y [M, N] from qa [M, K], sa [K/128, ld_sa],
    qw [N, K], sw [N/128, K/128].  Y is BF16 (fp8_blockscaled_gemm) or FP32
    (fp8_blockscaled_gemm_f32), following `y`'s dtype when y is given."""
    _require(qa, torch.uint8, "qa", 2)
    _require(qw, torch.uint8, "qw", 2)
    _require(sa, torch.float32, "sa", 2)
    M, K = qa.shape
    N = qw.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=qa.device)
    if y.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("y must be bfloat16 or float32")
    _require_min(y, y.dtype, "y", M, N)
    _require_min(qw, torch.uint8, "qw", N, K)
    _require_min(sa, torch.float32, "sa", K // 128, M)
    _require_count(sw, "sw", (N // 128) * (K // 128))
    fn = "fp8_blockscaled_gemm" if y.dtype == torch.bfloat16 else "fp8_blockscaled_gemm_f32"
    st = getattr(lib, fn)(_ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0), _ptr(qw), qw.stride(0), _ptr(sw),
                          _ptr(y), y.stride(0), M, N, K, _stream(stream))
    _check(fn, st)
    return y


def fp8_blockscaled_gemm_residual(qa, sa, qw, sw, residual, y=None, stream=None):
    """Y = bf16(FP32 block-scaled GEMM + residual), the residual (BF16 [M, N])
    added before the single output rounding.  y may be `residual` itself for
    an in-place update."""
    _require(qa, torch.uint8, "qa", 2)
    _require(qw, torch.uint8, "qw", 2)
    _require(sa, torch.float32, "sa", 2)
    _require(residual, torch.bfloat16, "residual", 2)
    M, K = qa.shape
    N = qw.shape[0]
    if tuple(residual.shape) != (M, N):
        raise ValueError("residual must be [M, N]")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=qa.device)
    _require_min(y, torch.bfloat16, "y", M, N)
    _require_min(qw, torch.uint8, "qw", N, K)
    _require_min(sa, torch.float32, "sa", K // 128, M)
    _require_count(sw, "sw", (N // 128) * (K // 128))
    st = lib.fp8_blockscaled_gemm_residual(_ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0), _ptr(qw), qw.stride(0),
                                           _ptr(sw), _ptr(residual), residual.stride(0), _ptr(y), y.stride(0),
                                           M, N, K, _stream(stream))
    _check("fp8_blockscaled_gemm_residual", st)
    return y


def fp8_blockscaled_gemm_workspace_bytes(M, N, K):
    """Bytes of split-K workspace that fp8_blockscaled_gemm takes from the
    library's pool for an M x N x K product on the current device (0: the
    shape's tiles are not split)."""
    out = ctypes.c_size_t(0)
    _check("fp8_blockscaled_gemm_workspace_bytes", lib.fp8_blockscaled_gemm_workspace_bytes(M, N, K, ctypes.byref(out)))
    return out.value


def fp8_blockscaled_gemm_noalloc(qa, sa, qw, sw, y=None, stream=None):
    """fp8_blockscaled_gemm (BF16 out) for callers that cannot allocate device
    memory: the split-K workspace lives in the library's fixed static device
    array instead of its memory pool, so the C call allocates nothing (this
    wrapper allocates y only when it is not given).  Calls share that array,
    so calls that could overlap on the GPU must be ordered (one stream)."""
    _require(qa, torch.uint8, "qa", 2)
    _require(qw, torch.uint8, "qw", 2)
    _require(sa, torch.float32, "sa", 2)
    M, K = qa.shape
    N = qw.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=qa.device)
    _require_min(y, torch.bfloat16, "y", M, N)
    _require_min(qw, torch.uint8, "qw", N, K)
    _require_min(sa, torch.float32, "sa", K // 128, M)
    _require_count(sw, "sw", (N // 128) * (K // 128))
    st = lib.fp8_blockscaled_gemm_noalloc(_ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0), _ptr(qw), qw.stride(0),
                                          _ptr(sw), _ptr(y), y.stride(0), M, N, K, _stream(stream))
    _check("fp8_blockscaled_gemm_noalloc", st)
    return y


def fp8_blockscaled_grouped_gemm(group_offsets, m_total, qa, sa, qw, sw, y=None, stream=None,
                                 out_dtype=torch.bfloat16):
    """Grouped GEMM: rows off[g]..off[g+1]-1 use expert g's weights.
    group_offsets: CUDA int32 [G+1]; m_total: host int equal to off[G];
    qw uint8 [G, N, K]; sw float32 [G, N/128, K/128].  Y is BF16 or FP32
    (following `y`'s dtype when given)."""
    if group_offsets.dtype != torch.int32 or not group_offsets.is_cuda or not group_offsets.is_contiguous():
        raise TypeError("group_offsets must be a contiguous CUDA int32 tensor")
    _require(qa, torch.uint8, "qa", 2)
    _require(sa, torch.float32, "sa", 2)
    if qw.dim() != 3 or not qw.is_contiguous() or not sw.is_contiguous():
        raise ValueError("qw [G, N, K] and sw [G, N/128, K/128] must be contiguous")
    G, N, K = qw.shape
    if y is None:
        y = torch.empty((m_total, N), dtype=out_dtype, device=qa.device)
    if y.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("y must be bfloat16 or float32")
    _require_min(y, y.dtype, "y", m_total, N)
    _require_min(qa, torch.uint8, "qa", m_total, K)
    _require_min(sa, torch.float32, "sa", K // 128, m_total)
    _require_count(sw, "sw", G * (N // 128) * (K // 128))
    if group_offsets.numel() != G + 1:
        raise ValueError("group_offsets must hold G + 1 offsets")
    fn = "fp8_blockscaled_grouped_gemm" if y.dtype == torch.bfloat16 else "fp8_blockscaled_grouped_gemm_f32"
    st = getattr(lib, fn)(G, _ptr(group_offsets), int(m_total), _ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0),
                          _ptr(qw), _ptr(sw), _ptr(y), y.stride(0), N, K, _stream(stream))
    _check(fn, st)
    return y


def fp8_dequant_weight_128x128(qw, sw, y=None, stream=None):
    """qw uint8 [N, K] (or [G, N, K]) + sw float32 [N/128, K/128] (or
    [G, N/128, K/128]) -> BF16 weights of the same shape."""
    if qw.dim() == 3:
        G, N, K = qw.shape
        y3 = y if y is not None else torch.empty((G, N, K), dtype=torch.bfloat16, device=qw.device)
        fp8_dequant_weight_128x128(qw.reshape(G * N, K), sw.reshape(G * N // 128, K // 128), y3.view(G * N, K),
                                   stream=stream)
        return y3
    _require(qw, torch.uint8, "qw", 2)
    N, K = qw.shape
    if y is None:
        y = torch.empty((N, K), dtype=torch.bfloat16, device=qw.device)
    _require_min(y, torch.bfloat16, "y", N, K)
    _require_count(sw, "sw", (N // 128) * (K // 128))
    st = lib.fp8_dequant_weight_128x128(_ptr(qw), N, K, qw.stride(0), _ptr(sw), _ptr(y), y.stride(0), _stream(stream))
    _check("fp8_dequant_weight_128x128", st)
    return y


def fp8_quant_act_1x128_t(x, qt=None, st=None, stream=None):
    """x bf16 [M, K] -> (qt uint8 [K, M] codes of x^T, st float32 [M/128, K]
    scales): 1x128 tiles of x^T.  M % 128 == 0."""
    _require(x, torch.bfloat16, "x", 2)
    M, K = x.shape
    if qt is None:
        qt = torch.empty((K, M), dtype=torch.uint8, device=x.device)
    if st is None:
        st = torch.empty((M // 128, ld_sa_for(K)), dtype=torch.float32, device=x.device)
    _require_min(qt, torch.uint8, "qt", K, M)
    _require_min(st, torch.float32, "st", M // 128, K)
    status = lib.fp8_quant_act_1x128_t(_ptr(x), M, K, x.stride(0), _ptr(qt), qt.stride(0), _ptr(st), st.stride(0),
                                       _stream(stream))
    _check("fp8_quant_act_1x128_t", status)
    return qt, st


def fp8_requant_act_1x128_t(qa, sa, qt=None, st=None, stream=None):
    """The FP8-cached activation (qa uint8 [M, K] 1x128 codes, sa float32
    [K/128, >=M] scales) -> (qt uint8 [K, M], st float32 [M/128, K]): each
    value dequantised to BF16, then 1x128 tiles of the transpose, as
    fp8_quant_act_1x128_t.  M % 128 == 0."""
    _require(qa, torch.uint8, "qa", 2)
    _require(sa, torch.float32, "sa", 2)
    M, K = qa.shape
    if qt is None:
        qt = torch.empty((K, M), dtype=torch.uint8, device=qa.device)
    if st is None:
        st = torch.empty((M // 128, ld_sa_for(K)), dtype=torch.float32, device=qa.device)
    _require_min(sa, torch.float32, "sa", K // 128, M)
    _require_min(qt, torch.uint8, "qt", K, M)
    _require_min(st, torch.float32, "st", M // 128, K)
    status = lib.fp8_requant_act_1x128_t(_ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0), M, K, _ptr(qt),
                                         qt.stride(0), _ptr(st), st.stride(0), _stream(stream))
    _check("fp8_requant_act_1x128_t", status)
    return qt, st


def fp8_pack_weight_128x128(qw, wp=None, stream=None):
    """qw uint8 [N, K] -> wp uint8 [N/128, K/128, 16384]: each 128x128 block
    as the 128-byte-swizzled image a GEMM stage holds (for
    fp8_blockscaled_gemm_packed)."""
    _require(qw, torch.uint8, "qw", 2)
    N, K = qw.shape
    if wp is None:
        wp = torch.empty((N // 128, K // 128, 128 * 128), dtype=torch.uint8, device=qw.device)
    if wp.dtype != torch.uint8 or not wp.is_contiguous() or wp.numel() != N * K:
        raise ValueError("wp must be a contiguous uint8 tensor of N*K bytes")
    _check("fp8_pack_weight_128x128", lib.fp8_pack_weight_128x128(_ptr(qw), N, K, qw.stride(0), _ptr(wp),
                                                                  _stream(stream)))
    return wp


def fp8_blockscaled_gemm_packed(qa, sa, wp, sw, y=None, stream=None):
    """fp8_blockscaled_gemm with B as packed tiles wp [N/128, K/128, 16384]
    (fp8_pack_weight_128x128); Y BF16 [M, N], bit for bit the same."""
    _require(qa, torch.uint8, "qa", 2)
    _require(sa, torch.float32, "sa", 2)
    if wp.dim() != 3 or wp.shape[2] != 128 * 128 or not wp.is_contiguous():
        raise ValueError("wp must be [N/128, K/128, 16384] contiguous")
    M, K = qa.shape
    N = wp.shape[0] * 128
    if wp.shape[1] * 128 != K:
        raise ValueError("wp and qa disagree on K")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=qa.device)
    _require_min(y, torch.bfloat16, "y", M, N)
    _require_min(sa, torch.float32, "sa", K // 128, M)
    _require_count(sw, "sw", (N // 128) * (K // 128))
    st = lib.fp8_blockscaled_gemm_packed(_ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0), _ptr(wp), _ptr(sw), _ptr(y),
                                         y.stride(0), M, N, K, _stream(stream))
    _check("fp8_blockscaled_gemm_packed", st)
    return y


def fp8_transpose_weight_128x128(qw, sw, qwt=None, swt=None, stream=None):
    """(qw uint8 [N, K], sw [N/128, K/128]) -> (qw^T [K, N], sw^T [K/128, N/128])."""
    _require(qw, torch.uint8, "qw", 2)
    N, K = qw.shape
    if qwt is None:
        qwt = torch.empty((K, N), dtype=torch.uint8, device=qw.device)
    if swt is None:
        swt = torch.empty((K // 128, N // 128), dtype=torch.float32, device=qw.device)
    _require_min(qwt, torch.uint8, "qwt", K, N)
    _require_count(sw, "sw", (N // 128) * (K // 128))
    _require_count(swt, "swt", (N // 128) * (K // 128))
    status = lib.fp8_transpose_weight_128x128(_ptr(qw), N, K, qw.stride(0), _ptr(sw), _ptr(qwt), qwt.stride(0),
                                              _ptr(swt), _stream(stream))
    _check("fp8_transpose_weight_128x128", status)
    return qwt, swt


def fp8_blockscaled_gemm_rowscaled(qa, sa, qb, sb, y=None, stream=None, out_dtype=torch.bfloat16):
    """Y [M, N] = sum_kb sa[kb, m] sb[kb, n] (chunk kb of dec(qa) dec(qb)^T):
    1x128 scales on both operands (the weight-gradient GEMM)."""
    _require(qa, torch.uint8, "qa", 2)
    _require(qb, torch.uint8, "qb", 2)
    _require(sa, torch.float32, "sa", 2)
    _require(sb, torch.float32, "sb", 2)
    M, K = qa.shape
    N = qb.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=qa.device)
    if y.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("y must be bfloat16 or float32")
    _require_min(y, y.dtype, "y", M, N)
    _require_min(qb, torch.uint8, "qb", N, K)
    _require_min(sa, torch.float32, "sa", K // 128, M)
    _require_min(sb, torch.float32, "sb", K // 128, N)
    fn = "fp8_blockscaled_gemm_rowscaled" if y.dtype == torch.bfloat16 else "fp8_blockscaled_gemm_rowscaled_f32"
    status = getattr(lib, fn)(_ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0), _ptr(qb), qb.stride(0), _ptr(sb),
                              sb.stride(0), _ptr(y), y.stride(0), M, N, K, _stream(stream))
    _check(fn, status)
    return y


def _codes_out(M, K, device):
    """A [M, K] code buffer whose row stride is K rounded up to 16 bytes (the
    C ABI's rule for FP8 row strides), so that K % 16 == 8 works too."""
    return torch.empty((M, (K + 15) // 16 * 16), dtype=torch.uint8, device=device)[:, :K]


def fp8_quant_per_token(x, q=None, s=None, stream=None):
    """x bf16 [M, K] -> (q uint8 [M, K], s float32 [M]): one scale per row.
    A q given by the caller needs a row stride that is a multiple of 16."""
    _require(x, torch.bfloat16, "x", 2)
    M, K = x.shape
    q = q if q is not None else _codes_out(M, K, x.device)
    s = s if s is not None else torch.empty((M,), dtype=torch.float32, device=x.device)
    _require_min(q, torch.uint8, "q", M, K)
    _require_count(s, "s", M)
    st = lib.fp8_quant_per_token(_ptr(x), M, K, x.stride(0), _ptr(q), q.stride(0), _ptr(s), _stream(stream))
    _check("fp8_quant_per_token", st)
    return q, s


def fp8_quant_per_channel(x, q=None, s=None, stream=None):
    """x bf16 [M, K] -> (q uint8 [M, K], s float32 [K]): one scale per column.
    A q given by the caller needs a row stride that is a multiple of 16."""
    _require(x, torch.bfloat16, "x", 2)
    M, K = x.shape
    q = q if q is not None else _codes_out(M, K, x.device)
    s = s if s is not None else torch.empty((K,), dtype=torch.float32, device=x.device)
    _require_min(q, torch.uint8, "q", M, K)
    _require_count(s, "s", K)
    st = lib.fp8_quant_per_channel(_ptr(x), M, K, x.stride(0), _ptr(q), q.stride(0), _ptr(s), _stream(stream))
    _check("fp8_quant_per_channel", st)
    return q, s


def e5m6_encode(x, codes=None, stream=None):
    """BF16 tensor (any shape, contiguous) -> E5M6 codes as int16 of the same shape."""
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or not x.is_cuda:
        raise TypeError("x must be a contiguous CUDA bfloat16 tensor")
    codes = codes if codes is not None else torch.empty(x.shape, dtype=torch.int16, device=x.device)
    _require_count(codes, "codes", x.numel(), dtype=torch.int16)
    st = lib.fp8bs_e5m6_encode_bf16(_ptr(x), x.numel(), _ptr(codes), _stream(stream))
    _check("fp8bs_e5m6_encode_bf16", st)
    return codes


def e5m6_decode(codes, y=None, stream=None):
    """E5M6 codes (int16, contiguous) -> BF16 values of the same shape (exact)."""
    if codes.dtype != torch.int16 or not codes.is_contiguous() or not codes.is_cuda:
        raise TypeError("codes must be a contiguous CUDA int16 tensor")
    y = y if y is not None else torch.empty(codes.shape, dtype=torch.bfloat16, device=codes.device)
    _require_count(y, "y", codes.numel(), dtype=torch.bfloat16)
    st = lib.fp8bs_e5m6_decode_bf16(_ptr(codes), codes.numel(), _ptr(y), _stream(stream))
    _check("fp8bs_e5m6_decode_bf16", st)
    return y


def fp8_swiglu_quant_act_1x128(gate_up, qa=None, sa=None, h=None, return_h=False, stream=None):
    """gate_up bf16 [M, 2F] (gate | up) -> (qa uint8 [M, F], sa float32 [F/128, ld_sa]) of
    h = bf16(silu(gate) * up); with return_h, also h (bf16 [M, F])."""
    _require(gate_up, torch.bfloat16, "gate_up", 2)
    M, F2 = gate_up.shape
    F = F2 // 2
    qa = qa if qa is not None else torch.empty((M, F), dtype=torch.uint8, device=gate_up.device)
    sa = sa if sa is not None else torch.empty((F // 128, ld_sa_for(M)), dtype=torch.float32, device=gate_up.device)
    if return_h and h is None:
        h = torch.empty((M, F), dtype=torch.bfloat16, device=gate_up.device)
    _require_min(qa, torch.uint8, "qa", M, F)
    _require_min(sa, torch.float32, "sa", F // 128, M)
    if h is not None:
        _require_min(h, torch.bfloat16, "h", M, F)
    st = lib.fp8_swiglu_quant_act_1x128(_ptr(gate_up), M, F, gate_up.stride(0), _ptr(qa), qa.stride(0), _ptr(sa),
                                        sa.stride(0), _ptr(h), h.stride(0) if h is not None else 0,
                                        _stream(stream))
    _check("fp8_swiglu_quant_act_1x128", st)
    return (qa, sa, h) if return_h else (qa, sa)


def linear_backward(x, w, dy, stream=None, grad_dtype=torch.float32, x_cache=None):
    """Both backward GEMMs of the FP8 linear layer, all in the library's
    kernels: dX = Q(dY) . Q(W)^T-blocks (BF16) and dW = Q(dY^T) . Q(X^T)^T
    (FP32 by default).  With x_cache = (qa, sa), the forward's 1x128 codes
    and scales of X, dW takes X from that FP8 cache
    (fp8_requant_act_1x128_t) and x may be None.  Returns (dx, dw)."""
    qw, sw = fp8_quant_weight_128x128(w, stream=stream)
    qwt, swt = fp8_transpose_weight_128x128(qw, sw, stream=stream)
    qdy, sdy = fp8_quant_act_1x128(dy, stream=stream)
    dx = fp8_blockscaled_gemm(qdy, sdy, qwt, swt, stream=stream)
    qdyt, sdyt = fp8_quant_act_1x128_t(dy, stream=stream)
    if x_cache is not None:
        qxt, sxt = fp8_requant_act_1x128_t(*x_cache, stream=stream)
    else:
        qxt, sxt = fp8_quant_act_1x128_t(x, stream=stream)
    dw = fp8_blockscaled_gemm_rowscaled(qdyt, sdyt, qxt, sxt, stream=stream, out_dtype=grad_dtype)
    return dx, dw


def fp8bs_last_device_error(stream=None):
    """Synchronise the stream and return (and clear) the device status code."""
    return lib.fp8bs_last_device_error(_stream(stream))


def fp8bs_set_wait_timeout_ns(ns: int):
    lib.fp8bs_set_wait_timeout_ns(int(ns))


def fp8bs_selftest_wait_timeout(ns: int, stream=None):
    _check("fp8bs_selftest_wait_timeout", lib.fp8bs_selftest_wait_timeout(int(ns), _stream(stream)))


def fp8bs_stream_timestamp(dst, index: int = 0, release_next: bool = False, stream=None):
    """Enqueue a device timestamp (ns) into dst[index] (an int64 CUDA tensor)
    once the work before it on the stream has completed; release_next lets
    the next kernel launch early, as fp8_quant_act_1x128 does."""
    if dst.dtype != torch.int64 or not dst.is_cuda or not 0 <= index < dst.numel():
        raise ValueError("dst must be an int64 CUDA tensor and index inside it")
    _check("fp8bs_stream_timestamp",
           lib.fp8bs_stream_timestamp(ctypes.c_void_p(dst.data_ptr() + 8 * index), int(bool(release_next)),
                                      _stream(stream)))


class HostPipeline:
    """The whole hot path on batches held in (pinned) host memory.

    Each submit() copies one batch (X, and W unless it is quantised once up
    front) host -> device, runs 1x128 activation quantisation, 128x128 weight
    quantisation and the block-scaled GEMM, and copies Y device -> host.  The
    three phases use three CUDA streams and `depth` sets of device buffers, so
    the copies of one batch overlap the kernels and copies of its neighbours.
    All arithmetic runs in the library's kernels; this class only owns
    buffers, streams, events and graphs.

    prequantised_w: a (qw, sw) pair already on the device (decode-style
    serving, where the weights stay resident); then only X moves per batch.

    use_graph: the kernels of each buffer set are captured once, at
    construction, into a CUDA graph that every submit replays (one launch
    instead of three C-ABI calls, which matters when the kernels are short).
    If the capture fails the calls are made directly, still on the GPU.
    """

    def __init__(self, M, N, K, device="cuda", depth=2, prequantised_w=None, use_graph=True):
        dev = torch.device(device)
        self.M, self.N, self.K, self.depth = M, N, K, depth
        self.h2d = torch.cuda.Stream(dev)
        self.compute = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.fixed_w = prequantised_w
        self.slots = []
        for _ in range(depth):
            slot = {
                "x": torch.zeros((M, K), dtype=torch.bfloat16, device=dev),
                "qa": torch.empty((M, K), dtype=torch.uint8, device=dev),
                "sa": torch.empty((K // 128, ld_sa_for(M)), dtype=torch.float32, device=dev),
                "y": torch.empty((M, N), dtype=torch.bfloat16, device=dev),
                "loaded": torch.cuda.Event(), "computed": torch.cuda.Event(), "stored": torch.cuda.Event(),
                "used": False, "graph": None,
            }
            if prequantised_w is None:
                slot["w"] = torch.zeros((N, K), dtype=torch.bfloat16, device=dev)
                slot["qw"] = torch.empty((N, K), dtype=torch.uint8, device=dev)
                slot["sw"] = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev)
            self.slots.append(slot)
        self.next = 0
        self.capture_error = None  # why the kernels are called directly, if capture failed
        if use_graph:
            self._capture_all(dev)

    def _compute(self, slot):
        """The slot's kernels, in order, on the compute stream."""
        fp8_quant_act_1x128(slot["x"], qa=slot["qa"], sa=slot["sa"], stream=self.compute)
        if self.fixed_w is None:
            fp8_quant_weight_128x128(slot["w"], qw=slot["qw"], sw=slot["sw"], stream=self.compute)
            qw, sw = slot["qw"], slot["sw"]
        else:
            qw, sw = self.fixed_w
        fp8_blockscaled_gemm(slot["qa"], slot["sa"], qw, sw, y=slot["y"], stream=self.compute)

    def _capture_all(self, dev):
        # one direct run per slot first: the library's per-device set-up
        # (synchronous runtime calls) must not happen inside a capture
        for slot in self.slots:
            self._compute(slot)
        torch.cuda.synchronize(dev)
        try:
            for slot in self.slots:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.compute, capture_error_mode="relaxed"):
                    self._compute(slot)
                slot["graph"] = g
        except Exception as e:  # e.g. a driver without the needed capture support
            torch.cuda.synchronize(dev)
            self.capture_error = f"{type(e).__name__}: {e}"
            for slot in self.slots:
                slot["graph"] = None

    @property
    def graphed(self):
        return all(slot["graph"] is not None for slot in self.slots)

    def submit(self, x_host, w_host, y_host):
        """Queue one batch; returns the event that completes when y_host holds Y."""
        slot = self.slots[self.next]
        self.next = (self.next + 1) % self.depth
        if slot["used"]:
            self.h2d.wait_event(slot["computed"])   # inputs of the slot's previous batch consumed
        with torch.cuda.stream(self.h2d):
            slot["x"].copy_(x_host, non_blocking=True)
            if self.fixed_w is None:
                slot["w"].copy_(w_host, non_blocking=True)
            slot["loaded"].record(self.h2d)
        self.compute.wait_event(slot["loaded"])
        if slot["used"]:
            self.compute.wait_event(slot["stored"])  # previous Y of the slot copied out
        if slot["graph"] is not None:
            with torch.cuda.stream(self.compute):
                slot["graph"].replay()
        else:
            self._compute(slot)
        slot["computed"].record(self.compute)
        self.d2h.wait_event(slot["computed"])
        with torch.cuda.stream(self.d2h):
            y_host.copy_(slot["y"], non_blocking=True)
            slot["stored"].record(self.d2h)
        slot["used"] = True
        return slot["stored"]

    def synchronize(self):
        for st in (self.h2d, self.compute, self.d2h):
            st.synchronize()


def linear_forward(x, w, stream=None):
    """The whole hot path: quantise x per 1x128 tile and w per 128x128 block,
    then the block-scaled GEMM.  Returns (y, (qa, sa, qw, sw))."""
    qa, sa = fp8_quant_act_1x128(x, stream=stream)
    qw, sw = fp8_quant_weight_128x128(w, stream=stream)
    return fp8_blockscaled_gemm(qa, sa, qw, sw, stream=stream), (qa, sa, qw, sw)
