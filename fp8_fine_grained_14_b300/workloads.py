"""Seeded synthetic inputs shaped like the DeepSeek-V3 projections.

This module holds no arithmetic of the method: it only draws inputs.  Both
the CUDA path and the CPU oracle consume what it returns, so the two are
compared on identical data.

Recipe (torch CPU generator, seed 0 unless stated, draws in this order:
X, then W, then any extras; FP32 normal draws, scaled, then rounded to BF16):
  tiny     X [128, 256] ~ N(0, 1);  W [256, 256] ~ N(0, 0.02)
  up       X [4096, 7168];          W [18432, 7168]     (hidden 7168 -> FFN 18432)
  down     X [4096, 18432] with 0.1 % of its channels (randperm(K)[:18])
           multiplied by 100 before the BF16 cast; W [7168, 18432]
  grouped  8192 tokens, each routed to 8 distinct experts of 64
           (multinomial without replacement over uniform weights);
           m_g = route counts, rows sorted by expert; X [65536, 7168];
           W [64, 2048, 7168]
  decode   X [64, 7168];            W [18432, 7168]
The hidden size 7168 and FFN size 18432 are the model's (CSDN article
"DeepSeek-V3：模型与权重全面解析", architecture list); 64 experts with top-8
routing shape the MoE case.  No dataset is involved.
"""
from __future__ import annotations

import torch

CONFIGS = {
    "tiny": dict(M=128, N=256, K=256),
    "up": dict(M=4096, N=18432, K=7168),
    "down": dict(M=4096, N=7168, K=18432, outlier_frac=0.001, outlier_scale=100.0),
    "grouped": dict(tokens=8192, topk=8, G=64, N=2048, K=7168),
    "decode": dict(M=64, N=18432, K=7168),
}


def gemm_flops(name: str) -> int:
    c = CONFIGS[name]
    if name == "grouped":
        return 2 * c["tokens"] * c["topk"] * c["N"] * c["K"]
    return 2 * c["M"] * c["N"] * c["K"]


def dense_inputs(M, N, K, seed=0, w_std=0.02, outlier_frac=0.0, outlier_scale=1.0):
    """X bf16 [M, K] ~ N(0, 1), W bf16 [N, K] ~ N(0, w_std), CPU tensors."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g, dtype=torch.float32)
    w = torch.randn(N, K, generator=g, dtype=torch.float32) * w_std
    n_out = int(outlier_frac * K)
    if n_out:
        idx = torch.randperm(K, generator=g)[:n_out]
        x[:, idx] *= outlier_scale
    return x.to(torch.bfloat16), w.to(torch.bfloat16)


def backward_inputs(M, N, K, seed=0, w_std=0.02, dy_std=1.0):
    """(x [M, K], w [N, K], dy [M, N]) BF16 CPU tensors for the backward GEMMs:
    X and W drawn as in dense_inputs, then the output gradient dY ~ N(0, dy_std)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g, dtype=torch.float32)
    w = torch.randn(N, K, generator=g, dtype=torch.float32) * w_std
    dy = torch.randn(M, N, generator=g, dtype=torch.float32) * dy_std
    return x.to(torch.bfloat16), w.to(torch.bfloat16), dy.to(torch.bfloat16)


def config_inputs(name: str, seed=0):
    """(x, w) for a dense configuration by name."""
    c = dict(CONFIGS[name])
    return dense_inputs(c.pop("M"), c.pop("N"), c.pop("K"), seed=seed, **c)


def grouped_inputs(tokens=8192, topk=8, G=64, N=2048, K=7168, seed=0, w_std=0.02):
    """(offsets int32 [G+1], x bf16 [tokens*topk, K], w bf16 [G, N, K]) on CPU."""
    g = torch.Generator().manual_seed(seed)
    rows = tokens * topk
    x = torch.randn(rows, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    w = (torch.randn(G, N, K, generator=g, dtype=torch.float32) * w_std).to(torch.bfloat16)
    routes = torch.multinomial(torch.ones(tokens, G), topk, replacement=False, generator=g)
    counts = torch.bincount(routes.flatten(), minlength=G)
    return grouped_offsets(counts), x, w


def grouped_offsets(counts):
    """int32 [G+1] prefix offsets of per-group row counts."""
    counts = torch.as_tensor(counts, dtype=torch.int64)
    off = torch.zeros(len(counts) + 1, dtype=torch.int32)
    off[1:] = torch.cumsum(counts, 0).to(torch.int32)
    return off
