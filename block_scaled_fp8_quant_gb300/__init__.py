"""block_scaled_fp8_quant_gb300 — block-scaled FP8 (W8A8) quant + GEMM for GB300.

Thin Python binding over the C ABI of ``libbfq.so`` (declared in
``include/bfq.h``).  Every step of the computation runs in the library's
sm_103a CUDA kernels; this module only marshals torch tensors (device
memory and the current stream) into the C calls.  There is no fallback: if
the library cannot be built or loaded, or a call returns a non-zero status,
a ``BfqError`` is raised.

Functions named like the C entry points (``bfq_quant``, ``bfq_gemm_block_fp8``,
...) take preallocated tensors; ``quant``, ``silu_mul_quant``,
``weight_block_quant``, ``gemm`` and ``gemm_masked`` allocate their outputs
with torch and call them.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

SCALE_F32 = 0
SCALE_F32_POW2 = 1
SCALE_UE8M0_PACKED = 2

STATUS_NAMES = {
    0: "BFQ_OK", 1: "BFQ_ERR_INVALID_ARG", 2: "BFQ_ERR_UNSUPPORTED_SHAPE",
    3: "BFQ_ERR_MISALIGNED", 4: "BFQ_ERR_FORMAT", 5: "BFQ_ERR_CUDA", 6: "BFQ_ERR_TIMEOUT",
    7: "BFQ_ERR_WORKSPACE", 8: "BFQ_ERR_DEVICE",
}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class BfqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)} ({status})")
        self.status = status


_debug = False


def library_path() -> str:
    return os.path.join(_HERE, "libbfq_debug.so" if _debug else "libbfq.so")


def load_library(build: bool = True, debug: bool | None = None):
    """Load libbfq.so (building it in-tree first when stale); raise if impossible.
    debug=True (before the first load of the process): libbfq_debug.so, the
    build whose kernels check their memory accesses against the arrays'
    extents and latch BFQ_ERR_DEVICE_BOUNDS (read by bfq_poll_device_status).
    debug=None: the library already loaded, else the release build."""
    global _lib, _debug
    with _lock:
        if _lib is not None:
            if debug is not None and debug != _debug:
                raise RuntimeError("the other build of the library is already loaded")
            return _lib
        _debug = bool(debug)
        if build:
            from . import _build

            _build.build(debug=_debug)
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libbfq.so not found at {path}: build the CUDA library first")
        lib = ctypes.CDLL(path)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "bfq_version": (I32, []),
            "bfq_status_string": (ctypes.c_char_p, [I32]),
            "bfq_quant": (I32, [P, I64, I64, I64, I32, I32, P, P, I64, P]),
            "bfq_silu_mul_quant": (I32, [P, I32, I32, I32, P, I32, P, P, I64, P]),
            "bfq_weight_block_quant": (I32, [P, I64, I64, I64, I32, P, P, P]),
            "bfq_gemm_workspace_bytes": (SZ, [I64, I64, I64, I32]),
            "bfq_gemm_block_fp8": (I32, [P, P, I32, I64, P, P, I64, I64, I64, P, P, SZ, P]),
            "bfq_gemm_block_fp8_masked": (I32, [P, P, I32, I64, P, P, P, I32, I32, I64, I64,
                                                I32, P, P, SZ, P]),
            "bfq_gemm_block_fp8_noalloc": (I32, [P, P, I32, I64, P, P, I64, I64, I64, P, P]),
            "bfq_gemm_block_fp8_quant": (I32, [P, P, I32, I64, P, P, I64, I64, I64, P, I32, P, P,
                                              I64, P, SZ, P]),
            "bfq_gemm_block_fp8_ue8m0": (I32, [P, P, I32, I64, P, P, I64, I64, I64, P, P]),
            "bfq_gemm_block_fp8_masked_ue8m0": (I32, [P, P, I32, I64, P, P, P, I32, I32, I64,
                                                      I64, P, P]),
            "bfq_interleave_gate_up": (I32, [P, P, I32, I64, I64, P, P, P]),
            "bfq_gemm_block_fp8_masked_silu_quant": (I32, [P, P, I32, I64, P, P, P, I32, I32, I64,
                                                          I64, I32, P, P, I64, P]),
            "bfq_gemm_block_fp8_masked_silu_quant_ue8m0": (I32, [P, P, I32, I64, P, P, P, I32,
                                                                I32, I64, I64, I32, P, P, I64,
                                                                P]),
            "bfq_gemm_noalloc_scratch_bytes": (SZ, []),
            "bfq_poll_device_status": (I32, [P]),
            "bfq_set_programmatic_launch": (I32, [I32]),
            "bfq_watchdog_selftest": (I32, [I32, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise BfqError(fn, status)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def align4(n: int) -> int:
    return (n + 3) // 4 * 4


def scale_cols(k: int, fmt: int) -> int:
    g = k // 128
    return (g + 3) // 4 if fmt == SCALE_UE8M0_PACKED else g


def scale_dtype(fmt: int) -> torch.dtype:
    return torch.int32 if fmt == SCALE_UE8M0_PACKED else torch.float32


# ---------------------------------------------------------------------------
# C-ABI mirrors (preallocated tensors)
# ---------------------------------------------------------------------------
def bfq_quant(x, q, scales, fmt: int, scale_ld: int, group: int = 128, stream=None) -> None:
    lib = load_library()
    M, K = x.shape
    _check("bfq_quant", lib.bfq_quant(_ptr(x), M, K, x.stride(0), group, fmt, _ptr(q),
                                      _ptr(scales), scale_ld, _stream(stream)))


def bfq_silu_mul_quant(x, valid_counts, q, scales, fmt: int, scale_ld: int,
                       stream=None) -> None:
    lib = load_library()
    E, T, two_i = x.shape
    assert x.is_contiguous() and q.is_contiguous()
    _check("bfq_silu_mul_quant",
           lib.bfq_silu_mul_quant(_ptr(x), E, T, two_i // 2, _ptr(valid_counts), fmt, _ptr(q),
                                  _ptr(scales), scale_ld, _stream(stream)))


def bfq_weight_block_quant(w, wq, sw, fmt: int, stream=None) -> None:
    lib = load_library()
    batch = 1 if w.dim() == 2 else w.shape[0]
    N, K = w.shape[-2:]
    assert w.is_contiguous() and wq.is_contiguous() and sw.is_contiguous()
    _check("bfq_weight_block_quant",
           lib.bfq_weight_block_quant(_ptr(w), batch, N, K, fmt, _ptr(wq), _ptr(sw),
                                      _stream(stream)))


def bfq_gemm_workspace_bytes(M: int, N: int, K: int, E: int = 0) -> int:
    return int(load_library().bfq_gemm_workspace_bytes(M, N, K, E))


def bfq_gemm_block_fp8(a_q, a_scales, a_fmt: int, a_scale_ld: int, w_q, w_scales, out,
                       workspace=None, stream=None) -> None:
    lib = load_library()
    M, K = a_q.shape
    N = w_q.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("bfq_gemm_block_fp8",
           lib.bfq_gemm_block_fp8(_ptr(a_q), _ptr(a_scales), a_fmt, a_scale_ld, _ptr(w_q),
                                  _ptr(w_scales), M, N, K, _ptr(out), _ptr(workspace), ws_bytes,
                                  _stream(stream)))


def bfq_gemm_block_fp8_quant(a_q, a_scales, a_fmt: int, a_scale_ld: int, w_q, w_scales, out,
                             q_fmt: int, q_out, q_scales, q_scale_ld: int, workspace=None,
                             stream=None) -> None:
    """GEMM whose epilogue also writes the 1 x 128 group quant of its bf16
    output (out may be None)."""
    lib = load_library()
    M, K = a_q.shape
    N = w_q.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("bfq_gemm_block_fp8_quant",
           lib.bfq_gemm_block_fp8_quant(_ptr(a_q), _ptr(a_scales), a_fmt, a_scale_ld, _ptr(w_q),
                                        _ptr(w_scales), M, N, K, _ptr(out), q_fmt, _ptr(q_out),
                                        _ptr(q_scales), q_scale_ld, _ptr(workspace), ws_bytes,
                                        _stream(stream)))


def gemm_quant(a_q, a_scales, a_fmt: int, w_q, w_scales, q_fmt: int, out=None, stream=None):
    """(q_out, q_scales) = 1 x 128 quant (format q_fmt) of the bf16 GEMM output,
    computed in the GEMM's epilogue; out (bf16 [M, N]) is also written when
    given."""
    M = a_q.shape[0]
    N = w_q.shape[0]
    q = torch.empty((M, N), dtype=torch.float8_e4m3fn, device=a_q.device)
    ld = align4(M)
    sc = torch.empty((scale_cols(N, q_fmt), ld), dtype=scale_dtype(q_fmt), device=a_q.device)
    ws = gemm_workspace(M, N, a_q.shape[1], a_q.device)
    bfq_gemm_block_fp8_quant(a_q, a_scales, a_fmt, a_scales.shape[-1], w_q, w_scales, out, q_fmt,
                             q, sc, ld, workspace=ws, stream=stream)
    return q, sc


def bfq_interleave_gate_up(w_q, w_scales, w_q_out, w_scales_out, stream=None) -> None:
    """[E, 2I, K] gate|up weight (and scales) -> 128-row blocks interleaved."""
    lib = load_library()
    E, N2, K = w_q.shape
    _check("bfq_interleave_gate_up",
           lib.bfq_interleave_gate_up(_ptr(w_q), _ptr(w_scales), E, N2 // 2, K, _ptr(w_q_out),
                                      _ptr(w_scales_out), _stream(stream)))


def interleave_gate_up(w_q, w_scales, stream=None):
    """Allocating form of bfq_interleave_gate_up."""
    w_o = torch.empty_like(w_q)
    s_o = torch.empty_like(w_scales)
    bfq_interleave_gate_up(w_q, w_scales, w_o, s_o, stream=stream)
    return w_o, s_o


def bfq_gemm_block_fp8_masked_silu_quant(a_q, a_scales, a_fmt: int, a_scale_ld: int, w_q,
                                         w_scales, valid_counts, q_fmt: int, q_out, q_scales,
                                         q_scale_ld: int, stream=None) -> None:
    """Masked up projection (interleaved weights) with silu-mul-quant fused."""
    lib = load_library()
    E, T, K = a_q.shape
    I = w_q.shape[1] // 2
    _check("bfq_gemm_block_fp8_masked_silu_quant",
           lib.bfq_gemm_block_fp8_masked_silu_quant(
               _ptr(a_q), _ptr(a_scales), a_fmt, a_scale_ld, _ptr(w_q), _ptr(w_scales),
               _ptr(valid_counts), E, T, I, K, q_fmt, _ptr(q_out), _ptr(q_scales), q_scale_ld,
               _stream(stream)))


def bfq_gemm_block_fp8_masked_silu_quant_ue8m0(a_q, a_scales, a_fmt: int, a_scale_ld: int, w_q,
                                               w_scales, valid_counts, q_fmt: int, q_out,
                                               q_scales, q_scale_ld: int, stream=None) -> None:
    """The fused up projection on the block-scaled kernel (UE8M0 scales)."""
    lib = load_library()
    E, T, K = a_q.shape
    I = w_q.shape[1] // 2
    _check("bfq_gemm_block_fp8_masked_silu_quant_ue8m0",
           lib.bfq_gemm_block_fp8_masked_silu_quant_ue8m0(
               _ptr(a_q), _ptr(a_scales), a_fmt, a_scale_ld, _ptr(w_q), _ptr(w_scales),
               _ptr(valid_counts), E, T, I, K, q_fmt, _ptr(q_out), _ptr(q_scales), q_scale_ld,
               _stream(stream)))


def gemm_masked_silu_quant(a_q, a_scales, a_fmt: int, w_q, w_scales, valid_counts, q_fmt: int,
                           stream=None):
    """(q [E, T, I], scales [E, cols, T]) of silu(gate) * up of the masked up
    projection; w_q / w_scales interleaved by interleave_gate_up."""
    E, T, _ = a_q.shape
    I = w_q.shape[1] // 2
    q = torch.empty((E, T, I), dtype=torch.float8_e4m3fn, device=a_q.device)
    sc = torch.empty((E, scale_cols(I, q_fmt), T), dtype=scale_dtype(q_fmt), device=a_q.device)
    bfq_gemm_block_fp8_masked_silu_quant(a_q, a_scales, a_fmt, a_scales.shape[-1], w_q, w_scales,
                                         valid_counts, q_fmt, q, sc, T, stream=stream)
    return q, sc


def bfq_gemm_block_fp8_noalloc(a_q, a_scales, a_fmt: int, a_scale_ld: int, w_q, w_scales, out,
                               stream=None) -> None:
    """bfq_gemm_block_fp8 without a workspace argument: for callers that may not
    allocate device memory (see include/bfq.h)."""
    lib = load_library()
    M, K = a_q.shape
    N = w_q.shape[0]
    _check("bfq_gemm_block_fp8_noalloc",
           lib.bfq_gemm_block_fp8_noalloc(_ptr(a_q), _ptr(a_scales), a_fmt, a_scale_ld,
                                          _ptr(w_q), _ptr(w_scales), M, N, K, _ptr(out),
                                          _stream(stream)))


def bfq_gemm_block_fp8_masked(a_q, a_scales, a_fmt: int, a_scale_ld: int, w_q, w_scales,
                              valid_counts, out, expected_m: int = 0, workspace=None,
                              stream=None) -> None:
    lib = load_library()
    E, T, K = a_q.shape
    N = w_q.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("bfq_gemm_block_fp8_masked",
           lib.bfq_gemm_block_fp8_masked(_ptr(a_q), _ptr(a_scales), a_fmt, a_scale_ld,
                                         _ptr(w_q), _ptr(w_scales), _ptr(valid_counts), E, T, N,
                                         K, expected_m, _ptr(out), _ptr(workspace), ws_bytes,
                                         _stream(stream)))


def bfq_gemm_block_fp8_ue8m0(a_q, a_scales, a_fmt: int, a_scale_ld: int, w_q, w_scales, out,
                             stream=None) -> None:
    """Dense GEMM for power-of-two scales on the tensor cores' block scaling."""
    lib = load_library()
    M, K = a_q.shape
    N = w_q.shape[0]
    _check("bfq_gemm_block_fp8_ue8m0",
           lib.bfq_gemm_block_fp8_ue8m0(_ptr(a_q), _ptr(a_scales), a_fmt, a_scale_ld, _ptr(w_q),
                                        _ptr(w_scales), M, N, K, _ptr(out), _stream(stream)))


def bfq_gemm_block_fp8_masked_ue8m0(a_q, a_scales, a_fmt: int, a_scale_ld: int, w_q, w_scales,
                                    valid_counts, out, stream=None) -> None:
    lib = load_library()
    E, T, K = a_q.shape
    N = w_q.shape[1]
    _check("bfq_gemm_block_fp8_masked_ue8m0",
           lib.bfq_gemm_block_fp8_masked_ue8m0(_ptr(a_q), _ptr(a_scales), a_fmt, a_scale_ld,
                                               _ptr(w_q), _ptr(w_scales), _ptr(valid_counts), E,
                                               T, N, K, _ptr(out), _stream(stream)))


def bfq_poll_device_status(stream=None) -> int:
    return int(load_library().bfq_poll_device_status(_stream(stream)))


def bfq_set_programmatic_launch(enable: bool) -> bool:
    """Switch programmatic dependent launch for later launches; returns the
    previous setting."""
    return bool(load_library().bfq_set_programmatic_launch(1 if enable else 0))


def bfq_watchdog_selftest(timeout_us: int, stream=None) -> None:
    _check("bfq_watchdog_selftest",
           load_library().bfq_watchdog_selftest(timeout_us, _stream(stream)))


# ---------------------------------------------------------------------------
# allocating helpers
# ---------------------------------------------------------------------------
def quant(x: torch.Tensor, fmt: int = SCALE_F32, scale_ld: int | None = None, stream=None):
    """bf16 [M, K] -> (e4m3 [M, K], column-major scales [cols, scale_ld])."""
    M, K = x.shape
    ld = align4(M) if scale_ld is None else scale_ld
    q = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=x.device)
    s = torch.empty((scale_cols(K, fmt), ld), dtype=scale_dtype(fmt), device=x.device)
    bfq_quant(x, q, s, fmt, ld, stream=stream)
    return q, s


def silu_mul_quant(x: torch.Tensor, valid_counts: torch.Tensor, fmt: int = SCALE_UE8M0_PACKED,
                   scale_ld: int | None = None, stream=None):
    """bf16 [E, T, 2I] -> (e4m3 [E, T, I], scales [E, cols, scale_ld]); padded rows untouched."""
    E, T, two_i = x.shape
    I = two_i // 2
    ld = align4(T) if scale_ld is None else scale_ld
    q = torch.empty((E, T, I), dtype=torch.float8_e4m3fn, device=x.device)
    s = torch.empty((E, scale_cols(I, fmt), ld), dtype=scale_dtype(fmt), device=x.device)
    bfq_silu_mul_quant(x, valid_counts, q, s, fmt, ld, stream=stream)
    return q, s


def weight_block_quant(w: torch.Tensor, fmt: int = SCALE_F32, stream=None):
    """bf16 [N, K] or [B, N, K] -> (e4m3 same shape, fp32 [.., ceil(N/128), K/128])."""
    N, K = w.shape[-2:]
    lead = tuple(w.shape[:-2])
    wq = torch.empty(w.shape, dtype=torch.float8_e4m3fn, device=w.device)
    sw = torch.empty(lead + ((N + 127) // 128, K // 128), dtype=torch.float32, device=w.device)
    bfq_weight_block_quant(w, wq, sw, fmt, stream=stream)
    return wq, sw


_ws_cache: dict = {}


def gemm_workspace(M: int, N: int, K: int, device) -> torch.Tensor | None:
    """Zero-initialised workspace sized for a dense (M, N, K) GEMM on `device`
    (one buffer per device, cached and grown on demand); None when the plan
    needs none.  Calls that share it must be ordered on one stream: the
    library keeps partial sums and per-tile counters in it during a call
    (and leaves the counters zero again)."""
    need = bfq_gemm_workspace_bytes(M, N, K)
    if need == 0:
        return None
    key = torch.device(device)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(need, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def gemm(a_q, a_scales, a_fmt: int, w_q, w_scales, out=None, workspace=None, stream=None):
    """out[M, N] (bf16) = block-scaled A * W^T."""
    M, K = a_q.shape
    N = w_q.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a_q.device)
    if workspace is None:
        workspace = gemm_workspace(M, N, K, a_q.device)
    bfq_gemm_block_fp8(a_q, a_scales, a_fmt, a_scales.shape[-1], w_q, w_scales, out,
                       workspace, stream=stream)
    return out


def gemm_ue8m0(a_q, a_scales, a_fmt: int, w_q, w_scales, out=None, stream=None):
    """out[M, N] (bf16) = block-scaled A * W^T for power-of-two scales, the
    scales applied by the MMA's block scaling."""
    M, K = a_q.shape
    N = w_q.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a_q.device)
    bfq_gemm_block_fp8_ue8m0(a_q, a_scales, a_fmt, a_scales.shape[-1], w_q, w_scales, out,
                             stream=stream)
    return out


def gemm_masked_ue8m0(a_q, a_scales, a_fmt: int, w_q, w_scales, valid_counts, out=None,
                      stream=None):
    """Masked form of gemm_ue8m0; rows r >= valid_counts[e] are not written."""
    E, T, K = a_q.shape
    N = w_q.shape[1]
    if out is None:
        out = torch.empty((E, T, N), dtype=torch.bfloat16, device=a_q.device)
    bfq_gemm_block_fp8_masked_ue8m0(a_q, a_scales, a_fmt, a_scales.shape[-1], w_q, w_scales,
                                    valid_counts, out, stream=stream)
    return out


def gemm_masked(a_q, a_scales, a_fmt: int, w_q, w_scales, valid_counts, out=None,
                expected_m: int = 0, stream=None):
    """out[E, T, N] (bf16); rows r >= valid_counts[e] are not written."""
    E, T, K = a_q.shape
    N = w_q.shape[1]
    if out is None:
        out = torch.empty((E, T, N), dtype=torch.bfloat16, device=a_q.device)
    bfq_gemm_block_fp8_masked(a_q, a_scales, a_fmt, a_scales.shape[-1], w_q, w_scales,
                              valid_counts, out, expected_m, stream=stream)
    return out
