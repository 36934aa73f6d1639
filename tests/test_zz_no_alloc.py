"""fp8_blockscaled_gemm_noalloc, the GEMM for callers that cannot allocate
device memory (an allocator they do not own, a step that must not
synchronise or fail on an allocation): its split-K workspace is the
library's fixed static device array instead of the memory pool.

Through the C ABI, two calls in a row must give exactly the result of
fp8_blockscaled_gemm, on shapes whose last round of tiles is split along K
(80 CTA-pair tiles on 74 resident pairs; the down-projection with 448) and on
one that is not, as fp8_blockscaled_gemm_workspace_bytes confirms before the
calls.  After a first call (the runtime may load the kernels' code then),
the device's free memory must not drop across the two calls.  This file
is collected last: the static array is state shared by every call on the
device."""
import ctypes

import pytest
import torch

import fp8_fine_grained_14_b300 as fb
from fp8_fine_grained_14_b300 import binding, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"
STATIC_SCRATCH_BYTES = 20 << 20  # the array's size, stated in include/fp8bs.h


def _noalloc(qa, sa, qw, sw, y):
    """One call of the entry point through the C ABI on the current stream."""
    M, K = qa.shape
    N = qw.shape[0]
    st = binding.lib.fp8_blockscaled_gemm_noalloc(
        ctypes.c_void_p(qa.data_ptr()), qa.stride(0), ctypes.c_void_p(sa.data_ptr()), sa.stride(0),
        ctypes.c_void_p(qw.data_ptr()), qw.stride(0), ctypes.c_void_p(sw.data_ptr()),
        ctypes.c_void_p(y.data_ptr()), y.stride(0), M, N, K,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, binding.Fp8bsError("fp8_blockscaled_gemm_noalloc", st)


@pytest.mark.parametrize("M,N,K,split", [(2048, 2560, 6144, True), (4096, 7168, 18432, True),
                                         (300, 512, 640, False)])
def test_noalloc_matches_gemm(M, N, K, split):
    need = fb.fp8_blockscaled_gemm_workspace_bytes(M, N, K)
    assert (need > 0) == split, need
    assert need <= STATIC_SCRATCH_BYTES
    x, w = workloads.dense_inputs(M, N, K, seed=M + N + 11 * K)
    qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    y1 = torch.full((M, N), 3.0, dtype=torch.bfloat16, device=DEV)
    y2 = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    y0 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    _noalloc(qa, sa, qw, sw, y0)  # first use: the runtime may load the kernels' code now
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    _noalloc(qa, sa, qw, sw, y1)
    _noalloc(qa, sa, qw, sw, y2)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert fb.fp8bs_last_device_error() == 0
    assert free_after >= free_before, (free_before, free_after)
    y_ref = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    torch.cuda.synchronize()
    assert torch.equal(y0, y_ref)
    assert torch.equal(y1, y_ref)
    assert torch.equal(y2, y_ref)
