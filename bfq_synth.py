"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws random numbers and nothing else: it holds none of the
quantization or GEMM arithmetic.  Both the CPU oracle and the CUDA library
consume what it produces.

Value distributions follow the workloads of "vLLM DeepGEMM FP8 Block GEMM
基准测试" §4.1/§4.4 (randn inputs, seed 42) widened to the activation
statistics of DeepSeek-style serving:

* activations: N(0, 1) fp32, 0.1 % of the entries (distinct positions drawn
  uniformly) multiplied by 50 in fp32, then rounded once to bf16 (RNE);
  optionally one whole 128-element group set to zero;
* weights: N(0, 0.02) fp32 rounded to bf16;
* per-expert valid counts: i.i.d. uniform on {0, ..., T_max};
* masked MoE inputs: rows r >= counts[e] are filled with NaN (a poison that
  any read of a padded row would spread).
"""
from __future__ import annotations

import torch

SEED = 42


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def activation(m: int, k: int, seed: int = SEED, outlier_frac: float = 1e-3,
               outlier_scale: float = 50.0, zero_group: bool = False,
               device: str | torch.device = "cpu") -> torch.Tensor:
    """bf16 [m, k] activation matrix."""
    g = _gen(seed, device)
    x = torch.randn((m, k), generator=g, device=device, dtype=torch.float32)
    numel = m * k
    n_out = int(outlier_frac * numel)
    if n_out > 0:
        if numel <= (1 << 24):
            idx = torch.randperm(numel, generator=g, device=device)[:n_out]
        else:  # distinct positions without materialising a full permutation
            idx = torch.randint(0, numel, (int(n_out * 1.01) + 16,), generator=g,
                                device=device).unique()[:n_out]
        flat = x.view(-1)
        flat[idx] = flat[idx] * outlier_scale
    if zero_group and k >= 128:
        r = int(torch.randint(0, m, (1,), generator=g, device=device).item())
        c = int(torch.randint(0, k // 128, (1,), generator=g, device=device).item())
        x[r, c * 128:(c + 1) * 128] = 0.0
    return x.to(torch.bfloat16)


def weight(n: int, k: int, seed: int = SEED + 1, std: float = 0.02,
           device: str | torch.device = "cpu") -> torch.Tensor:
    """bf16 [n, k] weight matrix, N(0, std)."""
    g = _gen(seed, device)
    w = torch.randn((n, k), generator=g, device=device, dtype=torch.float32) * std
    return w.to(torch.bfloat16)


def expert_weights(e: int, n: int, k: int, seed: int = SEED + 2, std: float = 0.02,
                   device: str | torch.device = "cpu") -> torch.Tensor:
    """bf16 [e, n, k] per-expert weights, N(0, std)."""
    g = _gen(seed, device)
    w = torch.randn((e, n, k), generator=g, device=device, dtype=torch.float32) * std
    return w.to(torch.bfloat16)


def valid_counts(e: int, t_max: int, seed: int = SEED + 3) -> torch.Tensor:
    """int32 [e] per-expert valid row counts ~ U{0..t_max} (CPU)."""
    g = _gen(seed, "cpu")
    return torch.randint(0, t_max + 1, (e,), generator=g, dtype=torch.int32)


def masked_activation(e: int, t_max: int, k: int, counts: torch.Tensor, seed: int = SEED + 4,
                      poison: bool = True, outlier_frac: float = 1e-3,
                      device: str | torch.device = "cpu") -> torch.Tensor:
    """bf16 [e, t_max, k]: activation rows per expert; rows >= counts[e] are NaN."""
    x = activation(e * t_max, k, seed=seed, outlier_frac=outlier_frac, device=device)
    x = x.view(e, t_max, k)
    if poison:
        rows = torch.arange(t_max, device=device).view(1, t_max)
        pad = rows >= counts.to(device).view(e, 1)
        x[pad] = float("nan")
    return x
