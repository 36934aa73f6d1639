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


def test_gemm_repeatable():
    """Two launches on the same inputs give bit-identical outputs."""
    x, w = workloads.dense_inputs(700, 1024, 1024, seed=8)
    y1, (qa, sa, qw, sw) = fb.linear_forward(x.to(DEV), w.to(DEV))
    y2 = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
