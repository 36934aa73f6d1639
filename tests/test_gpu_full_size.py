"""Full-size parity of the whole hot path on the benchmark's workloads.

Every activation code and scale, every weight code and scale, and every
output element of the up-projection, the down-projection with outlier
channels, the decode-shaped GEMM and the grouped MoE GEMM (64 experts,
65536 routed rows) is compared with the CPU oracle, run row-parallel over
the host's cores (oracle.parallel: the unchanged oracle on row slices).

Method: "The Definitive Information To Deepseek" -- 1x128 activation tiles and
128x128 weight blocks ("Figure 7 (a)", paragraph 3), online per-group scales
(paragraph 2), FP8 GEMM with per-chunk promotion and BF16 output
(paragraphs 1 and 4).  Codes and scales must be bit-exact; the GEMM output
must satisfy |y_gpu - y_ref| <= 1e-2 |y_ref| + 1e-3 rms(y_ref), with rms over
the whole output of the workload (for the grouped GEMM, the concatenated
sum(m_g) x N output).  The GPU runs each workload through the same entry
points, shapes and strides as the benchmark's timed step (the decode GEMM
both on plain and on packed weights).
"""
import numpy as np
import pytest
import torch

import fp8_fine_grained_14_b300 as fb
from fp8_fine_grained_14_b300 import workloads
from helpers import assert_codes_equal, assert_gemm_close_rows, assert_scales_equal, bf16_bits, f32, u8
from oracle.parallel import OraclePool

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pool():
    with OraclePool() as p:
        yield p


def _check_quant(pool, x, w2d, qa, sa, qw2d, sw2d, what):
    M = x.shape[0]
    qa_r, sa_r = pool.quant_act_1x128(bf16_bits(x))
    assert_codes_equal(u8(qa), qa_r, f"{what}: qa")
    assert_scales_equal(f32(sa)[:, :M], sa_r, f"{what}: sa")
    qw_r, sw_r = pool.quant_weight_128x128(bf16_bits(w2d))
    assert_codes_equal(u8(qw2d), qw_r, f"{what}: qw")
    assert_scales_equal(f32(sw2d), sw_r, f"{what}: sw")
    return qa_r, sa_r, qw_r, sw_r


@pytest.mark.parametrize("name", ["up", "down", "decode"])
def test_dense_full_size(pool, name):
    x, w = workloads.config_inputs(name)
    y, (qa, sa, qw, sw) = fb.linear_forward(x.to(DEV), w.to(DEV))
    y_packed = None
    if name == "decode":
        # the decode step streams weights packed before timing
        y_packed = fb.fp8_blockscaled_gemm_packed(qa, sa, fb.fp8_pack_weight_128x128(qw), sw).cpu()
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    y = y.cpu()
    qa_r, sa_r, qw_r, sw_r = _check_quant(pool, x, w, qa, sa, qw, sw, name)
    del qa, sa, qw, sw
    y_ref = pool.blockscaled_gemm(qa_r, sa_r, qw_r, sw_r)
    assert_gemm_close_rows(y, y_ref, what=name)
    if y_packed is not None:
        assert_gemm_close_rows(y_packed, y_ref, what=name + " (packed W)")
        assert torch.equal(y_packed, y), "packed-weight GEMM differs from the plain one"


def test_grouped_full_size(pool):
    c = workloads.CONFIGS["grouped"]
    offsets, x, w = workloads.grouped_inputs(**{k: c[k] for k in ("tokens", "topk", "G", "N", "K")})
    G, N, K = w.shape
    M = int(offsets[-1])
    xd, wd = x.to(DEV), w.to(DEV)
    qa, sa = fb.fp8_quant_act_1x128(xd)
    qw, sw = fb.fp8_quant_weight_128x128(wd)
    y = fb.fp8_blockscaled_grouped_gemm(offsets.to(DEV), M, qa, sa, qw, sw)
    torch.cuda.synchronize()
    assert fb.fp8bs_last_device_error() == 0
    del xd, wd
    y = y.cpu()
    counts = np.diff(offsets.numpy())
    assert counts.sum() == M and (counts > 0).all(), "every expert holds rows in this workload"
    qa_r, sa_r, qw_r, sw_r = _check_quant(pool, x, w.reshape(G * N, K), qa, sa, qw.reshape(G * N, K),
                                          sw.reshape(G * N // 128, K // 128), "grouped")
    del qa, sa, qw, sw
    y_ref = pool.blockscaled_grouped_gemm(offsets.numpy(), qa_r, sa_r, qw_r.reshape(G, N, K),
                                          sw_r.reshape(G, N // 128, K // 128))
    # every row of every expert (hence every 128-row tile of each) is compared,
    # against a tolerance whose rms is that of the whole concatenated output
    assert_gemm_close_rows(y, y_ref, what="grouped")
