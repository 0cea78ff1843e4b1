"""CPU oracle for block-scaled FP8 quantization and GEMM — TEST INFRASTRUCTURE.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it; the arithmetic lives in ``bfq_oracle.c`` (plain C,
built without fast-math or FP contraction) and this module only marshals
numpy arrays through ctypes.

Which definition each function follows (the pages and sections are listed in
the header of ``bfq_oracle.c``):

* ``e4m3_decode`` / ``e4m3_encode`` — OCP FP8 E4M3 ("fn") format,
  round-to-nearest-even, saturating.
* ``quant`` — per-token-group (1x128) quantization, "vLLM DeepGEMM FP8 Block
  GEMM 基准测试" §4.1 (``per_token_group_quant_fp8`` with column-major,
  TMA-aligned scales) and vLLM PR #29546 Purpose (UE8M0 scales packed four
  per uint32 inside the quant step).
* ``silu_mul_quant`` — vLLM PR #19885 Summary item 2 (fused silu-mul-quant
  that skips padded tokens).
* ``weight_block_quant`` — §4.1 ``per_block_cast_to_fp8`` (128x128 blocks,
  amax / fp8_max, optional ceil to a power of two).
* ``gemm`` / ``gemm_masked`` — §4.2 (per-K-block dot times a_s * b_s) and
  vLLM PR #19111 (masked per-expert grouped GEMM).

Every function is pinned by tests in ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

FMT_F32 = 0
FMT_F32_POW2 = 1
FMT_UE8M0_PACKED = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bfq_oracle.c")
_LIB = os.path.join(_HERE, "_bfq_oracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile bfq_oracle.c with gcc (IEEE fp32, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_oracle())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.orc_e4m3_decode.restype = ctypes.c_double
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
            lib.orc_expf.restype = ctypes.c_float
            lib.orc_expf.argtypes = [ctypes.c_float]
            lib.orc_silu.restype = ctypes.c_float
            lib.orc_silu.argtypes = [ctypes.c_float]
            lib.orc_quant.restype = I
            lib.orc_quant.argtypes = [P, I64, I64, I64, I, P, P, I64]
            lib.orc_silu_mul_quant.restype = I
            lib.orc_silu_mul_quant.argtypes = [P, I64, I64, I64, P, I, P, P, I64]
            lib.orc_weight_block_quant.restype = I
            lib.orc_weight_block_quant.argtypes = [P, I64, I64, I, P, P]
            lib.orc_gemm_rows.restype = I
            lib.orc_gemm_rows.argtypes = [P, P, I, I64, P, P, I64, I64, I64, P, I64, P]
            lib.orc_gemm_masked.restype = I
            lib.orc_gemm_masked.argtypes = [P, P, I, I64, P, P, P, I64, I64, I64, I64, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def align4(n: int) -> int:
    return (n + 3) // 4 * 4


def scale_cols(K: int, fmt: int) -> int:
    """Columns of the column-major scale array for K elements per row."""
    G = K // 128
    return (G + 3) // 4 if fmt == FMT_UE8M0_PACKED else G


def _scale_dtype(fmt: int):
    return np.uint32 if fmt == FMT_UE8M0_PACKED else np.float32


def bf16_bits(t) -> np.ndarray:
    """uint16 bit pattern of a bf16 torch tensor (CPU), as a numpy array."""
    import torch

    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# element functions
# --------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.orc_e4m3_decode(int(v)) for v in c], dtype=np.float64).reshape(
        np.shape(codes))


def e4m3_decode_table() -> np.ndarray:
    return e4m3_decode(np.arange(256, dtype=np.uint8))


def e4m3_encode(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, dtype=np.float32)
    flat = v.ravel()
    out = np.array([lib.orc_e4m3_encode(float(x)) for x in flat], dtype=np.uint8)
    return out.reshape(v.shape)


def expf(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, dtype=np.float32)
    return np.array([lib.orc_expf(float(x)) for x in v.ravel()], dtype=np.float32).reshape(
        v.shape)


def silu(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, dtype=np.float32)
    return np.array([lib.orc_silu(float(x)) for x in v.ravel()], dtype=np.float32).reshape(
        v.shape)


# --------------------------------------------------------------------------
# quantization
# --------------------------------------------------------------------------
def quant(x_bits: np.ndarray, fmt: int, scale_ld: int | None = None, scales_init=None):
    """Per-token-group quant of bf16 bits x[M][K] -> (q[M][K] uint8, scales).

    scales is [cols][scale_ld] (float32 or uint32 words), column-major over
    rows; scale_ld defaults to align4(M).  Entries of rows >= M are left as
    ``scales_init`` (zeros by default).
    """
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x.shape
    ld = align4(M) if scale_ld is None else scale_ld
    q = np.zeros((M, K), dtype=np.uint8)
    if scales_init is None:
        sc = np.zeros((scale_cols(K, fmt), ld), dtype=_scale_dtype(fmt))
    else:
        sc = np.ascontiguousarray(scales_init.copy(), dtype=_scale_dtype(fmt))
    rc = lib.orc_quant(_ptr(x), M, K, K, fmt, _ptr(q), _ptr(sc), ld)
    if rc:
        raise ValueError("oracle quant: bad arguments")
    return q, sc


def silu_mul_quant(x_bits: np.ndarray, counts, fmt: int, scale_ld: int | None = None,
                   q_init=None, scales_init=None):
    """x[E][T][2I] bf16 bits -> (q[E][T][I] uint8, scales[E][cols][ld]).

    Rows r >= counts[e] keep the values of ``q_init`` / ``scales_init``."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    E, T, two_i = x.shape
    I = two_i // 2
    ld = align4(T) if scale_ld is None else scale_ld
    cnt = np.ascontiguousarray(counts, dtype=np.int32)
    q = np.zeros((E, T, I), np.uint8) if q_init is None else np.ascontiguousarray(
        q_init.copy(), dtype=np.uint8)
    shape = (E, scale_cols(I, fmt), ld)
    sc = np.zeros(shape, _scale_dtype(fmt)) if scales_init is None else np.ascontiguousarray(
        scales_init.copy(), dtype=_scale_dtype(fmt))
    rc = lib.orc_silu_mul_quant(_ptr(x), E, T, I, _ptr(cnt), fmt, _ptr(q), _ptr(sc), ld)
    if rc:
        raise ValueError("oracle silu_mul_quant: bad arguments")
    return q, sc


def weight_block_quant(w_bits: np.ndarray, pow2: bool):
    """w[N][K] bf16 bits -> (wq[N][K] uint8, sw[ceil(N/128)][K/128] float32)."""
    lib = _load()
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    N, K = w.shape
    wq = np.zeros((N, K), np.uint8)
    sw = np.zeros(((N + 127) // 128, K // 128), np.float32)
    rc = lib.orc_weight_block_quant(_ptr(w), N, K, int(bool(pow2)), _ptr(wq), _ptr(sw))
    if rc:
        raise ValueError("oracle weight_block_quant: bad arguments")
    return wq, sw


# --------------------------------------------------------------------------
# GEMM
# --------------------------------------------------------------------------
def gemm(aq: np.ndarray, sa: np.ndarray, fmt_a: int, wq: np.ndarray, sw: np.ndarray,
         rows=None) -> np.ndarray:
    """fp64 C = A * W^T for the given rows of A (all rows by default)."""
    lib = _load()
    aq = np.ascontiguousarray(aq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=_scale_dtype(fmt_a))
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = aq.shape
    N, K2 = wq.shape
    assert K == K2
    r = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(
        rows, dtype=np.int64)
    out = np.zeros((len(r), N), np.float64)
    rc = lib.orc_gemm_rows(_ptr(aq), _ptr(sa), fmt_a, sa.shape[-1], _ptr(wq), _ptr(sw), M, N,
                           K, _ptr(r), len(r), _ptr(out))
    if rc:
        raise ValueError("oracle gemm: bad arguments")
    return out


def gemm_masked(aq: np.ndarray, sa: np.ndarray, fmt_a: int, wq: np.ndarray, sw: np.ndarray,
                counts) -> np.ndarray:
    """aq[E][T][K], wq[E][N][K] -> fp64 out[E][T][N]; rows >= counts[e] are NaN."""
    lib = _load()
    aq = np.ascontiguousarray(aq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=_scale_dtype(fmt_a))
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    cnt = np.ascontiguousarray(counts, dtype=np.int32)
    E, T, K = aq.shape
    _, N, _ = wq.shape
    out = np.full((E, T, N), np.nan, np.float64)
    rc = lib.orc_gemm_masked(_ptr(aq), _ptr(sa), fmt_a, sa.shape[-1], _ptr(wq), _ptr(sw),
                             _ptr(cnt), E, T, N, K, _ptr(out))
    if rc:
        raise ValueError("oracle gemm_masked: bad arguments")
    return out


def dequant_rows(q: np.ndarray, s: np.ndarray, fmt: int) -> np.ndarray:
    """fp64 values of quantized rows q[M][K] with column-major scales."""
    dec = e4m3_decode_table()
    M, K = q.shape
    vals = dec[q]
    G = K // 128
    out = np.empty((M, K), np.float64)
    for g in range(G):
        if fmt == FMT_UE8M0_PACKED:
            byte = (s[g // 4, :M].astype(np.uint64) >> np.uint64(8 * (g % 4))) & np.uint64(0xFF)
            sc = np.ldexp(1.0, byte.astype(np.int64) - 127)
        else:
            sc = s[g, :M].astype(np.float64)
        out[:, g * 128:(g + 1) * 128] = vals[:, g * 128:(g + 1) * 128] * sc[:, None]
    return out


def dequant_weight(wq: np.ndarray, sw: np.ndarray) -> np.ndarray:
    """fp64 values of 128x128 block-quantized weights."""
    dec = e4m3_decode_table()
    N, K = wq.shape
    vals = dec[wq]
    rep = np.repeat(np.repeat(sw.astype(np.float64), 128, axis=0), 128, axis=1)[:N, :K]
    return vals * rep
