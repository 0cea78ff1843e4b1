"""Helpers shared by the parity tests (no method arithmetic beyond norms)."""
import numpy as np
import torch

# The GEMM gate: |C_gpu - C_ref| <= 2e-3 * ||A_hat[m]|| * ||W_hat[n]||, where
# A_hat / W_hat are the dequantized operands the GEMM actually consumes and
# C_ref is the oracle's fp64 result.
GEMM_TOL = 2e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit pattern of a bf16 tensor (any device)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def codes(t: torch.Tensor) -> np.ndarray:
    """uint8 codes of an e4m3 tensor (any device)."""
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def scale_np(t: torch.Tensor, fmt: int) -> np.ndarray:
    a = t.detach().cpu().contiguous().numpy()
    return a.view(np.uint32) if fmt == 2 else a.view(np.float32)


def gemm_errors(out_gpu: np.ndarray, ref: np.ndarray, a_norms: np.ndarray,
                w_norms: np.ndarray):
    """(normalised error matrix, relative-to-value error matrix)."""
    denom = a_norms[:, None] * w_norms[None, :]
    diff = np.abs(out_gpu.astype(np.float64) - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        norm_err = np.where(denom > 0, diff / denom, diff)
    return norm_err, diff


def assert_gemm_close(out_gpu: np.ndarray, ref: np.ndarray, a_norms: np.ndarray,
                      w_norms: np.ndarray, what: str = "gemm"):
    assert out_gpu.shape == ref.shape, (out_gpu.shape, ref.shape)
    assert np.isfinite(out_gpu).all(), f"{what}: non-finite output"
    norm_err, diff = gemm_errors(out_gpu, ref, a_norms, w_norms)
    worst = float(norm_err.max()) if norm_err.size else 0.0
    assert worst <= GEMM_TOL, f"{what}: max normalised error {worst:.3e} > {GEMM_TOL}"
    # tighter sanity bound: bf16 rounding (2^-8 relative) plus fp32 accumulation
    slack = 2.0 ** -8 * np.abs(ref) + 1e-4 * a_norms[:, None] * w_norms[None, :]
    bad = diff > slack
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond 1 bf16 ulp + 1e-4 norm"
    return worst


def calc_diff(x: np.ndarray, y: np.ndarray) -> float:
    """1 - 2<x,y> / (|x|^2 + |y|^2) in fp64 ("vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.4)."""
    x = x.astype(np.float64)
    y = y.astype(np.float64)
    den = (x * x + y * y).sum()
    return float(1.0 - 2.0 * (x * y).sum() / den) if den > 0 else 0.0
