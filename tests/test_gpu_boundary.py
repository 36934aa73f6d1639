"""The C-ABI boundary on a GPU: no-op sizes, alignment errors, untouched
guard bands, and the bounded-wait failure path (a wait that nothing will
satisfy gives up, reports FP8BS_ERR_TIMEOUT and leaves the context usable)."""
import ctypes

import numpy as np
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
import oracle
from fp8_fine_grained_14_b300 import workloads
from fp8_fine_grained_14_b300.binding import lib
from helpers import assert_gemm_close, f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_m_zero_is_noop():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    qa, sa = fb.fp8_quant_act_1x128(x)
    assert qa.shape == (0, 256)
    qw, sw = fb.fp8_quant_weight_128x128(torch.zeros((128, 256), dtype=torch.bfloat16, device=DEV))
    y = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    assert y.shape == (0, 128)
    assert fb.fp8bs_last_device_error() == 0


def test_misaligned_pointers_rejected():
    buf = torch.zeros((4 * 256 + 16,), dtype=torch.bfloat16, device=DEV)
    q = torch.zeros((4 * 256 + 64,), dtype=torch.uint8, device=DEV)
    s = torch.zeros((64,), dtype=torch.float32, device=DEV)
    st = lib.fp8_quant_act_1x128(ctypes.c_void_p(buf.data_ptr() + 2), 4, 256, 256, ctypes.c_void_p(q.data_ptr()),
                                 256, ctypes.c_void_p(s.data_ptr()), 4, None)
    assert st == 2
    st = lib.fp8_quant_act_1x128(ctypes.c_void_p(buf.data_ptr()), 4, 256, 260, ctypes.c_void_p(q.data_ptr()),
                                 256, ctypes.c_void_p(s.data_ptr()), 4, None)
    assert st == 2
    st = lib.fp8_blockscaled_gemm(ctypes.c_void_p(q.data_ptr() + 8), 256, ctypes.c_void_p(s.data_ptr()), 4,
                                  ctypes.c_void_p(q.data_ptr()), 256, ctypes.c_void_p(s.data_ptr()),
                                  ctypes.c_void_p(buf.data_ptr()), 128, 2, 128, 256, None)
    assert st == 2


def test_quant_guard_bands():
    """Codes and scales are written only inside [M, K] / [K/128, M]."""
    M, K = 37, 384
    x, _ = workloads.dense_inputs(M, 128, K, seed=5)
    qa_buf = torch.full((M + 8, K), 0xA5, dtype=torch.uint8, device=DEV)
    sa_buf = torch.full((K // 128 + 1, 40), 9.0, dtype=torch.float32, device=DEV)
    fb.fp8_quant_act_1x128(x.to(DEV), qa=qa_buf[:M], sa=sa_buf[: K // 128])
    torch.cuda.synchronize()
    assert torch.all(qa_buf[M:] == 0xA5)
    assert torch.all(sa_buf[K // 128:] == 9.0) and torch.all(sa_buf[:, M:] == 9.0)


def test_wait_timeout_is_reported_and_context_survives():
    assert fb.fp8bs_last_device_error() == 0
    fb.fp8bs_selftest_wait_timeout(20_000_000)  # 20 ms limit
    assert fb.fp8bs_last_device_error() == 5    # FP8BS_ERR_TIMEOUT
    assert fb.fp8bs_last_device_error() == 0
    # the context is still usable: a normal GEMM runs and is correct
    x, w = workloads.dense_inputs(64, 256, 256, seed=3)
    y, _ = fb.linear_forward(x.to(DEV), w.to(DEV))
    y_ref, _ = oracle.linear_forward(f32(x), f32(w))
    assert_gemm_close(f32(y), y_ref)
    assert fb.fp8bs_last_device_error() == 0


def test_stream_timestamps_bracket_a_kernel():
    """Timestamps before and after a GEMM are ordered and span the kernel:
    the interval is positive and no longer than the host-observed wall time
    of the whole enqueue-and-synchronise."""
    import time

    x, w = workloads.dense_inputs(2048, 4096, 4096, seed=5)
    xd, wd = x.to(DEV), w.to(DEV)
    qa, sa = fb.fp8_quant_act_1x128(xd)
    qw, sw = fb.fp8_quant_weight_128x128(wd)
    t = torch.zeros(3, dtype=torch.int64, device=DEV)
    torch.cuda.synchronize()
    h0 = time.perf_counter_ns()
    fb.fp8bs_stream_timestamp(t, 0)
    fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    fb.fp8bs_stream_timestamp(t, 1)
    fb.fp8bs_stream_timestamp(t, 2)
    torch.cuda.synchronize()
    h1 = time.perf_counter_ns()
    t0, t1, t2 = t.tolist()
    assert 0 < t0 < t1 <= t2
    assert t1 - t0 < h1 - h0
    assert fb.fp8bs_last_device_error() == 0


def test_gemm_repeatable():
    """Two launches on the same inputs give bit-identical outputs."""
    x, w = workloads.dense_inputs(700, 1024, 1024, seed=8)
    y1, (qa, sa, qw, sw) = fb.linear_forward(x.to(DEV), w.to(DEV))
    y2 = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_empty_inputs_every_entry_point():
    """Zero rows (or zero elements) is a no-op for every entry point, and an
    expert group with no rows contributes nothing."""
    z = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    q, s = fb.fp8_quant_per_token(z)
    assert q.shape == (0, 256) and s.shape == (0,)
    q, s = fb.fp8_quant_per_channel(z)
    assert q.shape == (0, 256)
    qa, sa, h = fb.fp8_swiglu_quant_act_1x128(torch.empty((0, 512), dtype=torch.bfloat16, device=DEV), return_h=True)
    assert qa.shape == (0, 256) and h.shape == (0, 256)
    assert fb.e5m6_encode(torch.empty((0,), dtype=torch.bfloat16, device=DEV)).numel() == 0
    assert fb.e5m6_decode(torch.empty((0,), dtype=torch.int16, device=DEV)).numel() == 0
    qt, st = fb.fp8_quant_act_1x128_t(torch.empty((0, 256), dtype=torch.bfloat16, device=DEV))
    assert qt.shape == (256, 0)
    qa0, sa0 = fb.fp8_quant_act_1x128(z)
    qb, sb = fb.fp8_quant_act_1x128(torch.zeros((128, 256), dtype=torch.bfloat16, device=DEV))
    assert fb.fp8_blockscaled_gemm_rowscaled(qa0, sa0, qb, sb).shape == (0, 128)
    qw, sw = fb.fp8_quant_weight_128x128(torch.zeros((128, 256), dtype=torch.bfloat16, device=DEV))
    assert fb.fp8_blockscaled_gemm_noalloc(qa0, sa0, qw, sw).shape == (0, 128)
    # grouped: every group empty, and one empty group between two others
    off0 = torch.zeros((3,), dtype=torch.int32, device=DEV)
    qw3 = torch.zeros((2, 128, 256), dtype=torch.uint8, device=DEV)
    sw3 = torch.ones((2, 1, 2), dtype=torch.float32, device=DEV)
    assert fb.fp8_blockscaled_grouped_gemm(off0, 0, qa0, sa0, qw3, sw3).shape == (0, 128)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0


def test_grouped_empty_middle_group():
    """Three experts, the middle one with no rows: the other two match the
    dense oracle on their own rows."""
    g = torch.Generator().manual_seed(4)
    x = torch.randn(200, 256, generator=g).to(torch.bfloat16)
    w = (torch.randn(3, 128, 256, generator=g) * 0.02).to(torch.bfloat16)
    offsets = torch.tensor([0, 120, 120, 200], dtype=torch.int32)
    qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
    qw, sw = fb.fp8_quant_weight_128x128(w.reshape(384, 256).to(DEV))
    y = fb.fp8_blockscaled_grouped_gemm(offsets.to(DEV), 200, qa, sa, qw.reshape(3, 128, 256), sw.reshape(3, 1, 2))
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    qa_r, sa_r = oracle.quant_act_1x128(f32(x))
    parts = []
    for gi, (r0, r1) in enumerate([(0, 120), (120, 120), (120, 200)]):
        if r1 == r0:
            continue
        qw_r, sw_r = oracle.quant_weight_128x128(f32(w[gi]))
        parts.append(oracle.blockscaled_gemm(qa_r[r0:r1], sa_r[:, r0:r1], qw_r, sw_r))
    assert_gemm_close(f32(y), np.concatenate(parts))


def test_wrappers_reject_undersized_buffers():
    """The C ABI sees only pointers and row strides, so the Python wrappers
    check that every buffer they pass holds the rows, columns or scales the
    call will touch, and raise before anything is launched."""
    x = torch.zeros((256, 256), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        fb.fp8_quant_act_1x128(x, qa=torch.empty((128, 256), dtype=torch.uint8, device=DEV))
    with pytest.raises(ValueError):
        fb.fp8_quant_act_1x128(x, sa=torch.empty((2, 128), dtype=torch.float32, device=DEV))
    qa, sa = fb.fp8_quant_act_1x128(x)
    qw, sw = fb.fp8_quant_weight_128x128(x)
    with pytest.raises(ValueError):
        fb.fp8_blockscaled_gemm(qa, sa, qw, sw[:1].contiguous())
    with pytest.raises(ValueError):
        fb.fp8_blockscaled_gemm(qa, sa, qw, sw, y=torch.empty((256, 128), dtype=torch.bfloat16, device=DEV))
    with pytest.raises(ValueError):
        fb.fp8_blockscaled_gemm_residual(qa, sa, qw, sw, torch.zeros((256, 256), dtype=torch.bfloat16, device=DEV),
                                         y=torch.empty((200, 256), dtype=torch.bfloat16, device=DEV))
    with pytest.raises(ValueError):
        fb.fp8_transpose_weight_128x128(qw, sw, swt=torch.empty((1, 1), dtype=torch.float32, device=DEV))
    with pytest.raises(ValueError):
        fb.fp8_dequant_weight_128x128(qw, sw[:1].contiguous())
    qw3 = qw.reshape(2, 128, 256)
    sw3 = sw.reshape(2, 1, 2)
    with pytest.raises(ValueError):
        fb.fp8_blockscaled_grouped_gemm(torch.zeros((2,), dtype=torch.int32, device=DEV), 256, qa, sa, qw3, sw3)
    with pytest.raises(ValueError):
        fb.fp8_blockscaled_grouped_gemm(torch.zeros((3,), dtype=torch.int32, device=DEV), 300, qa, sa, qw3, sw3)
    with pytest.raises(ValueError):
        fb.fp8_requant_act_1x128_t(qa, sa, st=torch.empty((1, 256), dtype=torch.float32, device=DEV))
    with pytest.raises(ValueError):
        fb.fp8_quant_per_token(x, s=torch.empty((100,), dtype=torch.float32, device=DEV))
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
