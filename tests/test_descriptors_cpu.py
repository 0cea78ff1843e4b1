"""Tensor-core descriptor encodings, checked on the CPU before any kernel
that uses them runs.

A host program built from the kernels' own header prints the instruction
descriptors of tcgen05.mma .kind::f8f6f4 (e4m3 x e4m3 -> fp32) and
.kind::mxf8f6f4.block_scale (UE8M0 scale factors, scale byte 0..3) and the
shared-memory descriptors of the swizzled operand tiles and of the
tcgen05.cp scale-factor source.  Each field is decoded here from the bit
positions of the PTX ISA's tcgen05 "Instruction descriptor" and "Shared
memory descriptor" tables and compared with what the kernels intend: a
wrong format, major-ness, dimension, scale type or layout would otherwise
only show on the GPU, possibly as an illegal-instruction fault."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_scaled_fp8_quant_gb300", "csrc")

_PROGRAM = r"""
#include <stdio.h>
#include "bfq_device.cuh"
int main() {
  printf("f8f6f4 %u\n", bfq::idesc_e4m3_f32(128, 256));
  printf("f8f6f4_n128 %u\n", bfq::idesc_e4m3_f32(128, 128));
  for (unsigned b = 0; b < 4; ++b) printf("bs%u %u\n", b, bfq::idesc_e4m3_bs(128, 256, b));
  printf("sw128 %llu\n", (unsigned long long)bfq::sdesc_kmajor_sw128(0x12400u));
  printf("rows16 %llu\n", (unsigned long long)bfq::sdesc_rows16(0x1C830u));
  return 0;
}
"""


def _field(v, lo, hi):
    return (v >> lo) & ((1 << (hi - lo)) - 1)


@pytest.fixture(scope="module")
def values(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    d = tmp_path_factory.mktemp("desc")
    src = d / "desc.cu"
    src.write_text(_PROGRAM)
    exe = d / "desc"
    subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr",
                    "-I", os.path.join(ROOT, "include"), "-I", CSRC, str(src), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return {k: int(v) for k, v in (line.split() for line in out.splitlines())}


def _common_mma_fields(v, M, N):
    assert _field(v, 0, 2) == 0, "sparsity selector"
    assert _field(v, 2, 3) == 0, "dense"
    assert _field(v, 7, 10) == 0, "A format e4m3"
    assert _field(v, 10, 13) == 0, "B format e4m3"
    assert _field(v, 13, 14) == 0 and _field(v, 14, 15) == 0, "no negation"
    assert _field(v, 15, 16) == 0 and _field(v, 16, 17) == 0, "A and B K-major"
    assert _field(v, 17, 23) == N >> 3, "N >> 3"
    assert _field(v, 24, 29) == M >> 4, "M >> 4"


@pytest.mark.parametrize("key,N", [("f8f6f4", 256), ("f8f6f4_n128", 128)])
def test_f8f6f4_instruction_descriptor(values, key, N):
    v = values[key]
    _common_mma_fields(v, 128, N)
    assert _field(v, 3, 4) == 0, "no saturation"
    assert _field(v, 4, 6) == 1, "D format f32"
    assert _field(v, 6, 7) == 0 and _field(v, 23, 24) == 0 and _field(v, 29, 30) == 0
    assert _field(v, 30, 32) == 0, "no max shift"


@pytest.mark.parametrize("byte", [0, 1, 2, 3])
def test_block_scaled_instruction_descriptor(values, byte):
    v = values[f"bs{byte}"]
    _common_mma_fields(v, 128, 256)
    assert _field(v, 3, 4) == 0 and _field(v, 6, 7) == 0 and _field(v, 31, 32) == 0
    assert _field(v, 4, 6) == byte, "B scale-factor byte"
    assert _field(v, 29, 31) == byte, "A scale-factor byte"
    assert _field(v, 23, 24) == 1, "scale factors UE8M0"


def test_swizzled_operand_descriptor(values):
    v = values["sw128"]
    assert _field(v, 0, 14) << 4 == 0x12400, "start address"
    assert _field(v, 32, 46) << 4 == 1024, "8-row swizzle atoms 1024 bytes apart"
    assert _field(v, 46, 48) == 1, "descriptor version"
    assert _field(v, 49, 52) == 0, "base offset (1024-aligned tiles)"
    assert _field(v, 52, 53) == 0, "relative leading byte offset"
    assert _field(v, 61, 64) == 2, "128-byte swizzle"


def test_scale_factor_copy_source_descriptor(values):
    v = values["rows16"]
    assert _field(v, 0, 14) << 4 == 0x1C830, "start address"
    assert _field(v, 16, 30) == 0, "one core matrix along K"
    assert _field(v, 32, 46) << 4 == 128, "8-row x 16-byte core matrices contiguous"
    assert _field(v, 46, 48) == 1, "descriptor version"
    assert _field(v, 49, 53) == 0
    assert _field(v, 61, 64) == 0, "no swizzle"
