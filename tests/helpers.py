"""Shared helpers for the parity tests: host conversions, the GEMM
acceptance rule and sampled comparisons.  The CUDA path is reached only
through the package's C-ABI binding; the oracle only through `oracle`."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# GEMM acceptance: |y_gpu - y_ref| <= REL * |y_ref| + ABS_RMS * rms(y_ref),
# rms over the whole output tensor of the case.  The BF16 output rounding
# alone contributes up to 2^-9 relative; FP32 chunk accumulation in tensor
# memory and FP32 promotion contribute far less.
REL = 1e-2
ABS_RMS = 1e-3


def f32(t: torch.Tensor) -> np.ndarray:
    """BF16/FP32 torch tensor -> float32 numpy (exact for BF16)."""
    return t.detach().to("cpu", torch.float32).numpy()


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.uint8)


def assert_gemm_close(y_gpu, y_ref, rms=None, what="gemm"):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y_gpu.shape == y_ref.shape, (y_gpu.shape, y_ref.shape)
    if rms is None:
        rms = float(np.sqrt(np.mean(y_ref * y_ref))) if y_ref.size else 0.0
    err = np.abs(y_gpu - y_ref)
    tol = REL * np.abs(y_ref) + ABS_RMS * rms
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)
        worst = np.unravel_index(np.argmax(err - tol), err.shape)
        rows = np.unique(idx[:, 0])
        cols = np.unique(idx[:, 1])
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; rows {rows[:8]}.. ({rows.size}), "
            f"cols {cols[:8]}.. ({cols.size}); worst at {worst}: gpu={y_gpu[worst]!r} ref={y_ref[worst]!r}; "
            f"rms={rms:.4g}")


def assert_gemm_close_rows(y_gpu, y_ref, rows_per_chunk=4096, what="gemm"):
    """assert_gemm_close over a large output, in row chunks (bounded host
    memory), with rms taken over the WHOLE reference output."""
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert tuple(y_gpu.shape) == y_ref.shape, (tuple(y_gpu.shape), y_ref.shape)
    rms = float(np.sqrt(np.mean(np.square(y_ref)))) if y_ref.size else 0.0
    for r0 in range(0, y_ref.shape[0], rows_per_chunk):
        r1 = min(y_ref.shape[0], r0 + rows_per_chunk)
        assert_gemm_close(f32(y_gpu[r0:r1]), y_ref[r0:r1], rms=rms, what=f"{what} rows {r0}..{r1 - 1}")
    return rms


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw BF16 bit patterns of a CPU BF16 tensor (what the row-parallel
    oracle takes, at half the size of float32 values)."""
    return t.contiguous().view(torch.int16).numpy()


def assert_codes_equal(got, want, what):
    got = np.asarray(got, dtype=np.uint8)
    want = np.asarray(want, dtype=np.uint8)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.argwhere(got != want)
    assert bad.size == 0, (f"{what}: {len(bad)} codes differ, first at {bad[:4].tolist()}: "
                           f"gpu={[hex(int(got[tuple(b)])) for b in bad[:4]]} "
                           f"oracle={[hex(int(want[tuple(b)])) for b in bad[:4]]}")


def assert_scales_equal(got, want, what):
    got = np.ascontiguousarray(got, dtype=np.float32)
    want = np.ascontiguousarray(want, dtype=np.float32)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.argwhere(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, (f"{what}: {len(bad)} scales differ, first at {bad[:4].tolist()}: "
                           f"gpu={[float(got[tuple(b)]) for b in bad[:4]]} "
                           f"oracle={[float(want[tuple(b)]) for b in bad[:4]]}")


def sample_rows(M, n, seed=0):
    """Sorted sample of distinct row indices touching every 128-row tile:
    about n rows spread evenly over the tiles (drawn without replacement),
    always including the first and last row; every row when M <= n."""
    if M <= n:
        return np.arange(M, dtype=np.int64)
    rng = np.random.default_rng(seed)
    tiles = (M + 127) // 128
    per = max(1, n // max(tiles, 1))
    rows = set([0, M - 1])
    for t in range(tiles):
        lo, hi = t * 128, min(M, t * 128 + 128)
        rows.update((lo + rng.choice(hi - lo, size=min(per, hi - lo), replace=False)).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def sample_blocks(NB, n, seed=0):
    """Sorted sample of n weight block-rows including the first and last."""
    rng = np.random.default_rng(seed)
    pick = set([0, NB - 1])
    pick.update(rng.choice(NB, size=min(n, NB), replace=False).tolist())
    return np.array(sorted(pick), dtype=np.int64)


def oracle_dense_sampled(x_cpu, w_cpu, rows, nblocks):
    """Oracle quantisation + GEMM restricted to `rows` of X and to the 128-row
    weight blocks `nblocks` (every output column of those blocks).  Rows are
    independent under 1x128 quantisation and whole blocks are independent
    under 128x128 quantisation, so the restriction is exact.
    Returns (qa_rows, sa_rows [KB, len(rows)], qw_blocks, sw_blocks, y_ref, cols)."""
    x = f32(x_cpu)[rows]
    wrows = np.concatenate([np.arange(b * 128, b * 128 + 128) for b in nblocks])
    w = f32(w_cpu)[wrows]
    qa, sa = oracle.quant_act_1x128(x)
    qw, sw = oracle.quant_weight_128x128(w)
    y = oracle.blockscaled_gemm(qa, sa, qw, sw)
    return qa, sa, qw, sw, y, wrows
