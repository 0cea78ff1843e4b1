"""Fused silu-and-mul + quant over a masked per-expert batch on the GPU vs the
oracle ("[EP+DP] Optimize the little operations in the DeepGEMM + DeepEP low
latency case", Summary item 2): codes and scales bit-exact for valid rows,
padded rows neither read (NaN poison never spreads) nor written (sentinels
survive)."""
import numpy as np
import pytest
import torch

import bfq_synth as synth
from helpers import bits, codes, scale_np

pytestmark = pytest.mark.gpu

Q_SENT = 0xAB


def _run(bfq, x, counts, fmt, ld):
    E, T, two_i = x.shape
    I = two_i // 2
    q = torch.full((E, T, I), Q_SENT, dtype=torch.uint8, device="cuda").view(
        torch.float8_e4m3fn)
    sc = torch.empty((E, bfq.scale_cols(I, fmt), ld), dtype=bfq.scale_dtype(fmt), device="cuda")
    sc.fill_(int(np.uint32(0xDEADBEEF).view(np.int32)) if fmt == 2 else -7.0)
    bfq.bfq_silu_mul_quant(x.cuda(), counts.cuda(), q, sc, fmt, ld)
    torch.cuda.synchronize()
    return q, sc


def _check(orc, x, counts, q, sc, fmt):
    E, T, two_i = x.shape
    oq, osc = orc.silu_mul_quant(bits(x), counts.numpy(), fmt, scale_ld=sc.shape[-1])
    qh = codes(q)
    sh = scale_np(sc, fmt)
    sent = np.uint32(0xDEADBEEF) if fmt == 2 else np.float32(-7.0)
    for e in range(E):
        c = max(0, min(int(counts[e]), T))
        assert np.array_equal(qh[e, :c], oq[e, :c]), f"expert {e} codes"
        assert np.array_equal(sh[e, :, :c], osc[e, :, :c]), f"expert {e} scales"
        assert np.all(qh[e, c:] == Q_SENT), f"expert {e}: padded rows written"
        assert np.all(sh[e, :, c:] == sent), f"expert {e}: padded scales written"


def test_silu_mul_quant_moe_config(cuda_lib, orc):
    """E = 32, T_max = 256, 2I = 4096, counts ~ U{0..256}, padded rows NaN."""
    bfq = cuda_lib
    E, T, I = 32, 256, 2048
    counts = synth.valid_counts(E, T)
    x = synth.masked_activation(E, T, 2 * I, counts)
    q, sc = _run(bfq, x, counts, 2, T)
    _check(orc, x, counts, q, sc, 2)


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_silu_mul_quant_edges(cuda_lib, orc, fmt):
    bfq = cuda_lib
    E, T, I = 5, 20, 640  # I/128 = 5 groups: a partial packed word
    counts = torch.tensor([0, 20, 1, 13, -3], dtype=torch.int32)
    x = synth.masked_activation(E, T, 2 * I, counts.clamp(min=0), seed=5)
    q, sc = _run(bfq, x, counts, fmt, 24)
    _check(orc, x, counts, q, sc, fmt)


def test_silu_mul_quant_large_activations(cuda_lib, orc):
    """Gate values up to +-300 drive exp to 0 and to overflow."""
    bfq = cuda_lib
    E, T, I = 2, 8, 256
    counts = torch.tensor([8, 5], dtype=torch.int32)
    g = torch.Generator().manual_seed(9)
    x = (torch.randn(E, T, 2 * I, generator=g) * 100).to(torch.bfloat16)
    q, sc = _run(bfq, x, counts, 2, 8)
    _check(orc, x, counts, q, sc, 2)


@pytest.mark.parametrize("fmt", [0, 2])
def test_silu_mul_quant_many_experts(cuda_lib, orc, fmt):
    """More experts than the walk over valid units holds counts for (1100 >
    1024): the per-block form, one block per pair of rows of an expert."""
    bfq = cuda_lib
    E, T, I = 1100, 3, 256
    g = torch.Generator().manual_seed(17)
    counts = torch.randint(0, T + 1, (E,), generator=g, dtype=torch.int32)
    x = synth.masked_activation(E, T, 2 * I, counts, seed=18)
    q, sc = _run(bfq, x, counts, fmt, 4)
    _check(orc, x, counts, q, sc, fmt)


def test_silu_mul_quant_gate_binades_in_order(cuda_lib, orc):
    """Every bf16 gate below 2^100 in magnitude, in bit-pattern order, with
    up = 1: each 128-group holds one binade of one sign and y is silu(g)
    itself, so a wrong table entry shows in its group's codes far more often
    than with random up values (tests/test_silu_table_gpu.py covers every
    pattern, NaN included, that way)."""
    bfq = cuda_lib
    pats = np.arange(65536, dtype=np.uint32)
    pats = pats[((pats >> 7) & 0xFF) < 227].astype(np.uint16)
    I = 2048
    T = -(-len(pats) // I)
    gate = np.full(T * I, 0x3F80, np.uint16)  # 1.0 after the last pattern
    gate[:len(pats)] = pats
    x = torch.empty((1, T, 2 * I), dtype=torch.bfloat16)
    x[0, :, :I] = torch.from_numpy(gate.view(np.int16)).view(torch.bfloat16).reshape(T, I)
    x[0, :, I:] = 1.0
    counts = torch.tensor([T], dtype=torch.int32)
    ld = -(-T // 4) * 4
    for fmt in (0, 2):
        q, sc = _run(bfq, x, counts, fmt, ld)
        _check(orc, x, counts, q, sc, fmt)


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_silu_mul_quant_large_batch_edges(cuda_lib, orc, fmt):
    """A batch of many rows per expert (thousands of blocks) with a partial
    packed word (I/128 = 5 groups), empty experts, a count past T_max and a
    negative one, padded rows NaN."""
    bfq = cuda_lib
    E, T, I = 8, 400, 640
    counts = torch.tensor([0, 400, 1, 399, -3, 517, 250, 0], dtype=torch.int32)
    x = synth.masked_activation(E, T, 2 * I, counts.clamp(0, T), seed=31)
    q, sc = _run(bfq, x, counts, fmt, 400)
    _check(orc, x, counts, q, sc, fmt)


@pytest.mark.parametrize("fmt", [0, 2])
def test_silu_mul_quant_thousand_small_experts(cuda_lib, orc, fmt):
    """1000 experts of at most 4 rows, most rows padded."""
    bfq = cuda_lib
    E, T, I = 1000, 4, 256
    g = torch.Generator().manual_seed(41)
    counts = torch.randint(0, T + 1, (E,), generator=g, dtype=torch.int32)
    x = synth.masked_activation(E, T, 2 * I, counts, seed=42)
    q, sc = _run(bfq, x, counts, fmt, 4)
    _check(orc, x, counts, q, sc, fmt)
