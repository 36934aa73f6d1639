"""fp8_blockscaled_gemm_noalloc: the block-scaled GEMM with its split-K
workspace in the library's fixed static device array.  On shapes whose last
round of tiles is split along K (80 CTA-pair tiles on 74 resident pairs; the
down-projection with 448 tiles) and on one that is not split, two calls give
exactly the result of fp8_blockscaled_gemm.  This file runs last: the static
array is shared state of the device."""
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
from fp8_fine_grained_14_b300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("M,N,K", [(2048, 2560, 6144), (4096, 7168, 18432), (300, 512, 640)])
def test_noalloc_matches_gemm(M, N, K):
    x, w = workloads.dense_inputs(M, N, K, seed=M + N + 11 * K)
    qa, sa = fb.fp8_quant_act_1x128(x.to(DEV))
    qw, sw = fb.fp8_quant_weight_128x128(w.to(DEV))
    y_ref = fb.fp8_blockscaled_gemm(qa, sa, qw, sw)
    y1 = fb.fp8_blockscaled_gemm_noalloc(qa, sa, qw, sw)
    y2 = torch.full_like(y1, 7.0)
    fb.fp8_blockscaled_gemm_noalloc(qa, sa, qw, sw, y=y2)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    assert torch.equal(y1, y_ref)
    assert torch.equal(y2, y_ref)
