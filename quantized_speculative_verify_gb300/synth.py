"""Seeded synthetic inputs for the verify-pass linear layer.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no rotation, no quantization, no GEMM).  Both the CUDA
path and the CPU oracle receive the same arrays from here.

Distributions (the workload shapes of the 9B-class verify pass; the pages
measure on a real checkpoint and prompt, which these stand in for):
  weights      N(0, 0.02) fp32, a given fraction of uniformly chosen entries
               multiplied by 20 (outliers);
  activations  N(0, 1) fp32, optionally a few whole input channels multiplied
               by 30, or a fraction of entries replaced by Student-t(nu=3)
               draws (heavy tail).
All draws come from torch.Generator streams seeded explicitly, on the device
the tensors are made on.
"""
from __future__ import annotations

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def weights(N: int, K: int, seed: int, outlier_frac: float = 0.005, outlier_mult: float = 20.0,
            std: float = 0.02, device="cpu") -> torch.Tensor:
    """W [N][K] fp32 ~ N(0, std) with round(outlier_frac * N * K) entries scaled by outlier_mult."""
    g = _gen(seed, device)
    W = torch.randn((N, K), generator=g, device=device, dtype=torch.float32).mul_(std)
    n_out = int(round(outlier_frac * N * K))
    if n_out > 0:
        idx = torch.randperm(N * K, generator=g, device=device)[:n_out]
        W.view(-1)[idx] *= outlier_mult
    return W


def activations(M: int, K: int, seed: int, outlier_channels: int = 0, channel_mult: float = 30.0,
                heavy_frac: float = 0.0, nu: int = 3, device="cpu") -> torch.Tensor:
    """X [M][K] fp32 ~ N(0, 1); `outlier_channels` uniformly chosen columns x channel_mult in every
    row; round(heavy_frac * M * K) uniformly chosen entries replaced by Student-t(nu) draws."""
    g = _gen(seed, device)
    X = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    if outlier_channels > 0:
        cols = torch.randperm(K, generator=g, device=device)[:outlier_channels]
        X[:, cols] *= channel_mult
    n_heavy = int(round(heavy_frac * M * K))
    if n_heavy > 0:
        idx = torch.randperm(M * K, generator=g, device=device)[:n_heavy]
        z = torch.randn(n_heavy, generator=g, device=device, dtype=torch.float64)
        chi2 = torch.randn((n_heavy, nu), generator=g, device=device, dtype=torch.float64).pow(2).sum(1)
        t = z / torch.sqrt(chi2 / nu)
        X.view(-1)[idx] = t.to(torch.float32)
    return X


# The five workloads of the verify pass.  `x` gives the activation recipe,
# `w` the weight recipe; `layers` lists (name, K, N) for the whole-pass case.
CONFIGS = {
    "tiny_256": dict(K=256, N=256, Ms=(1, 16), fmt="w4", G=32, seed=0,
                     w=dict(outlier_frac=0.005), x=dict(outlier_channels=2)),
    "attn_4096": dict(K=4096, N=4096, Ms=(16,), fmt="w4", G=64, seed=1,
                      w=dict(outlier_frac=0.001), x=dict(outlier_channels=2)),
    "gateup_w8": dict(K=4096, N=2 * 12288, Ms=(1, 4, 16, 32), fmt="w8", G=128, seed=2,
                      w=dict(outlier_frac=0.005), x=dict(heavy_frac=0.01)),
    "sweep_8192_w8": dict(K=8192, N=8192, Ms=(1, 2, 4, 8, 16, 32, 64, 128), fmt="w8", G=128, seed=3,
                          w=dict(outlier_frac=0.005), x=dict()),
    "sweep_8192_w4": dict(K=8192, N=8192, Ms=(1, 2, 4, 8, 16, 32, 64, 128), fmt="w4", G=64, seed=3,
                          w=dict(outlier_frac=0.005), x=dict()),
}

# 9B-class decoder: 32 layers of q/k/v/o, fused gate+up and down, plus the LM head.
DECODER_9B = dict(n_layers=32, hidden=4096, kv=1024, ffn=12288, vocab=151552, fmt="w4", G=64, M=16, seed=4,
                  w=dict(outlier_frac=0.005), x=dict(outlier_channels=2))


def decoder_linears(cfg=DECODER_9B, fuse_qkv: bool = False):
    """(name, K, N) of every linear of one verify pass, in launch order."""
    h, kv, f = cfg["hidden"], cfg["kv"], cfg["ffn"]
    out = []
    for l in range(cfg["n_layers"]):
        if fuse_qkv:
            out.append((f"l{l}.qkv", h, h + 2 * kv))
        else:
            out += [(f"l{l}.q", h, h), (f"l{l}.k", h, kv), (f"l{l}.v", h, kv)]
        out += [(f"l{l}.o", h, h), (f"l{l}.gate_up", h, 2 * f), (f"l{l}.down", f, h)]
    out.append(("lm_head", h, cfg["vocab"]))
    return out


def decoder_gemms(cfg=DECODER_9B, fuse_qkv: bool = True):
    """The GEMMs of one verify pass in launch order: (name, K, parts) with
    parts = [(part name, N, weight seed index)].  q, k and v read the same
    activations and, with fuse_qkv, run as one GEMM over their three weight
    matrices; gate and up always run as one GEMM over their two.  The seed
    index of a part is its position in the unfused list of matrices."""
    h, kv, f = cfg["hidden"], cfg["kv"], cfg["ffn"]
    out, idx = [], 0
    for l in range(cfg["n_layers"]):
        qkv = [(f"l{l}.q", h, idx), (f"l{l}.k", kv, idx + 1), (f"l{l}.v", kv, idx + 2)]
        if fuse_qkv:
            out.append((f"l{l}.qkv", h, qkv))
        else:
            out += [(name, h, [(name, n, i)]) for name, n, i in qkv]
        out.append((f"l{l}.o", h, [(f"l{l}.o", h, idx + 3)]))
        out.append((f"l{l}.gate_up", h, [(f"l{l}.gate", f, idx + 4), (f"l{l}.up", f, idx + 5)]))
        out.append((f"l{l}.down", f, [(f"l{l}.down", h, idx + 6)]))
        idx += 7
    out.append(("lm_head", h, [("lm_head", cfg["vocab"], idx)]))
    return out


def decoder_weight_count(cfg=DECODER_9B) -> int:
    return sum(K * N for _, K, N in decoder_linears(cfg))


def layer_seed(base: int, index: int) -> int:
    return base * 1000 + index

