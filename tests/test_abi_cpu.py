"""The C ABI without a GPU: the library builds, loads and exports every symbol
declared in include/bfq.h, and host-side validation rejects bad arguments
before any CUDA call is made."""
import ctypes
import os
import re

import pytest

import block_scaled_fp8_quant_gb300 as bfq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bfq.h")

OK, INVALID, SHAPE, MISALIGNED, FORMAT, CUDA = 0, 1, 2, 3, 4, 5
A16 = 0x10000  # a 16-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module")
def lib():
    return bfq.load_library()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bfq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("bfq_quant", "bfq_silu_mul_quant", "bfq_gemm_block_fp8",
              "bfq_gemm_block_fp8_masked", "bfq_weight_block_quant"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    assert lib.bfq_version() >= 10000
    assert lib.bfq_status_string(0) == b"BFQ_OK"
    assert lib.bfq_status_string(6) == b"BFQ_ERR_TIMEOUT"
    assert lib.bfq_status_string(999) == b"BFQ_ERR_UNKNOWN"


def test_quant_validation(lib):
    q = lib.bfq_quant
    assert q(A16, 4, 100, 100, 128, 0, A16, A16, 4, None) == SHAPE       # K % 128
    assert q(A16, 4, 256, 256, 64, 0, A16, A16, 4, None) == SHAPE        # group != 128
    assert q(A16, 4, 256, 256, 128, 7, A16, A16, 4, None) == INVALID     # bad format
    assert q(A16, 4, 256, 128, 128, 0, A16, A16, 4, None) == INVALID     # ld_x < K
    assert q(A16, 8, 256, 256, 128, 0, A16, A16, 4, None) == INVALID     # scale_ld < M
    assert q(None, 4, 256, 256, 128, 0, A16, A16, 4, None) == INVALID    # null x
    assert q(A16 + 2, 4, 256, 256, 128, 0, A16, A16, 4, None) == MISALIGNED
    assert q(A16, 4, 256, 260, 128, 0, A16, A16, 4, None) == MISALIGNED  # row stride
    assert q(A16, 4, 256, 256, 128, 2, A16, A16, 6, None) == MISALIGNED  # scale_ld % 4
    assert q(A16, 4, 256, 256, 128, 0, A16, A16, 5, None) == MISALIGNED
    assert q(A16, 0, 256, 256, 128, 0, None, None, 0, None) == OK        # empty: no-op


def test_silu_mul_quant_validation(lib):
    f = lib.bfq_silu_mul_quant
    assert f(A16, 2, 16, 100, A16, 2, A16, A16, 16, None) == SHAPE      # I % 128
    assert f(A16, 2, 16, 256, A16, 2, A16, A16, 8, None) == INVALID     # scale_ld < T
    assert f(A16, 2, 16, 256, None, 2, A16, A16, 16, None) == INVALID   # null counts
    assert f(A16 + 8, 2, 16, 256, A16, 2, A16, A16, 16, None) == MISALIGNED
    assert f(A16, 2, 16, 256, A16, 2, A16, A16, 18, None) == MISALIGNED  # scale_ld % 4
    assert f(A16, 0, 16, 256, None, 2, None, None, 16, None) == OK      # no experts


def test_weight_quant_validation(lib):
    f = lib.bfq_weight_block_quant
    assert f(A16, 1, 256, 100, 0, A16, A16, None) == SHAPE
    assert f(A16, 1, 256, 256, 2, A16, A16, None) == FORMAT            # packed weights
    assert f(A16, 0, 256, 256, 0, A16, A16, None) == INVALID
    assert f(A16 + 4, 1, 256, 256, 0, A16, A16, None) == MISALIGNED


def test_gemm_validation(lib):
    g = lib.bfq_gemm_block_fp8
    assert g(A16, A16, 0, 8, A16, A16, 8, 100, 256, A16, None, 0, None) == SHAPE  # N % 64
    assert g(A16, A16, 0, 8, A16, A16, 8, 128, 200, A16, None, 0, None) == SHAPE  # K % 128
    assert g(A16, A16, 0, 4, A16, A16, 8, 128, 256, A16, None, 0, None) == INVALID  # ld < M
    assert g(A16, A16, 9, 8, A16, A16, 8, 128, 256, A16, None, 0, None) == INVALID  # format
    assert g(A16, A16, 0, 8, A16, A16, 8, 128, 256, None, None, 0, None) == INVALID
    assert g(A16 + 1, A16, 0, 8, A16, A16, 8, 128, 256, A16, None, 0, None) == MISALIGNED
    assert g(A16, A16, 0, 10, A16, A16, 8, 128, 256, A16, None, 0, None) == MISALIGNED
    assert g(A16, A16, 0, 8, A16, A16, 8, 128, 256, A16, None, 64, None) == INVALID  # ws null
    assert g(A16, A16, 0, 0, A16, A16, 0, 128, 256, A16, None, 0, None) == OK        # M = 0
    m = lib.bfq_gemm_block_fp8_masked
    assert m(A16, A16, 2, 16, A16, A16, A16, 2, 16, 100, 256, 0, A16, None, 0, None) == SHAPE
    assert m(A16, A16, 2, 8, A16, A16, A16, 2, 16, 128, 256, 0, A16, None, 0, None) == INVALID
    assert m(A16, A16, 2, 16, A16, A16, None, 2, 16, 128, 256, 0, A16, None, 0, None) == INVALID
    assert m(A16, A16, 2, 16, A16, A16, A16, 0, 16, 128, 256, 0, A16, None, 0, None) == OK


def test_watchdog_selftest_validation(lib):
    assert lib.bfq_watchdog_selftest(0, None) == INVALID
    assert lib.bfq_watchdog_selftest(2000000, None) == INVALID


def test_valid_call_without_gpu_reports_cuda_error(lib):
    """On a machine without a GPU a well-formed call fails cleanly (no CPU path)."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("this machine has a GPU")
    assert lib.bfq_quant(A16, 4, 256, 256, 128, 0, A16, A16, 4, None) == CUDA
    assert lib.bfq_gemm_workspace_bytes(8, 4096, 7168, 0) == 0


def test_workspace_bytes_are_zero(lib):
    """Every split reduces through distributed shared memory: no plan, dense
    (E = 0) or masked (E >= 1), needs a workspace."""
    ws = lib.bfq_gemm_workspace_bytes
    for m, n, k, e in [(8, 4096, 7168, 0), (64, 32768, 512, 0), (4096, 4096, 7168, 0),
                       (256, 4096, 7168, 32)]:
        assert ws(m, n, k, e) == 0


def test_programmatic_launch_switch(lib):
    """The process-wide PDL switch returns the previous setting (default on)."""
    assert lib.bfq_set_programmatic_launch(0) == 1
    assert lib.bfq_set_programmatic_launch(0) == 0
    assert lib.bfq_set_programmatic_launch(5) == 0   # any non-zero value means on
    assert lib.bfq_set_programmatic_launch(1) == 1
