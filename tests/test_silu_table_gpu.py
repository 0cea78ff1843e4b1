"""silu by table lookup in the fused silu-and-mul + quant ("[EP+DP] Optimize
the little operations in the DeepGEMM + DeepEP low latency case", Summary
item 2).  The gate is bf16, so silu has 65536 possible inputs; the library
evaluates its silu once per device for all of them and looks it up.  The
table path must give the oracle's codes and scales bit for bit for every
finite gate value (and NaN), and the kernel that computes silu (used while a graph is being
captured before the table exists) must give the same bits as the table."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from helpers import bits, codes, scale_np

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _all_gates_input(seed):
    """x [1, 32, 2 * 2048] bf16: the gate half holds each of the 65536 bf16 bit
    patterns once (NaN included), except that the two infinities are zeros,
    and the up half seeded values in (-1, 1), so that no group's amax is
    infinite (a group with an infinite amax has no finite scale; the pages
    do not define that case)."""
    I = 2048
    codes16 = torch.arange(65536, dtype=torch.int32)
    codes16[0x7F80] = 0x0000  # +inf -> +0
    codes16[0xFF80] = 0x8000  # -inf -> -0
    gates = codes16.to(torch.int16).view(torch.bfloat16)
    g = torch.Generator().manual_seed(seed)
    up = (torch.rand(65536, generator=g) * 1.98 - 0.99).to(torch.bfloat16)
    x = torch.empty((1, 32, 2 * I), dtype=torch.bfloat16)
    x[0, :, :I] = gates.view(32, I)
    x[0, :, I:] = up.view(32, I)
    return x


@pytest.mark.parametrize("fmt", [0, 2])
def test_every_bf16_gate_matches_the_oracle(cuda_lib, orc, fmt):
    bfq = cuda_lib
    x = _all_gates_input(seed=11 + fmt)
    counts = torch.tensor([32], dtype=torch.int32)
    q, sc = bfq.silu_mul_quant(x.cuda(), counts.cuda(), fmt)
    torch.cuda.synchronize()
    oq, osc = orc.silu_mul_quant(bits(x), counts.numpy(), fmt, scale_ld=sc.shape[-1])
    assert np.array_equal(codes(q), oq)
    assert np.array_equal(scale_np(sc, fmt), osc)


_SCRIPT = r"""
import sys
sys.path.insert(0, sys.argv[1])
import torch
import block_scaled_fp8_quant_gb300 as bfq
sys.path.insert(0, sys.argv[1] + "/tests")
from test_silu_table_gpu import _all_gates_input
bfq.load_library()
x = _all_gates_input(seed=5).cuda()
counts = torch.tensor([32], dtype=torch.int32, device="cuda")
I = 2048
q_g = torch.empty((1, 32, I), dtype=torch.float8_e4m3fn, device="cuda")
s_g = torch.empty((1, 4, 32), dtype=torch.int32, device="cuda")
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g):  # the first silu call of this process: no table yet
    bfq.bfq_silu_mul_quant(x, counts, q_g, s_g, 2, 32)
g.replay()
torch.cuda.synchronize()
q_t, s_t = bfq.silu_mul_quant(x, counts, 2)  # builds the table, looks silu up
torch.cuda.synchronize()
same = torch.equal(q_g.view(torch.uint8), q_t.view(torch.uint8)) and torch.equal(s_g, s_t)
print("SAME" if same else "DIFFERENT")
"""


def test_computed_silu_equals_table_silu(cuda_lib):
    """In a fresh process, silu_mul_quant captured into a graph before any
    eager call (the kernel computes silu), then eagerly (table lookup)."""
    r = subprocess.run([sys.executable, "-c", _SCRIPT, ROOT], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.strip().splitlines()[-1] == "SAME"
