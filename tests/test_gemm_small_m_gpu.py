"""Dense block-scaled FP8 GEMM with few activation rows (M <= 128) on the GPU
vs the oracle ("vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.2 for the GEMM,
§4.3/§五 for why small m is its own case: the weight bytes are the cost).

With one row tile, the launch plan splits K over the CTAs of a thread-block
cluster (fewer output tiles than SMs) and adds the fp32 partials in split
order through distributed shared memory, or walks more tiles than SMs with
one CTA per SM.  Every checked element is within 2e-3 * ||A_hat[m]|| *
||W_hat[n]|| of the oracle's fp64 result (plus the one-bf16-ulp sanity
bound); results are deterministic."""
import numpy as np
import pytest
import torch

import bfq_synth as synth
from helpers import assert_gemm_close, bits, calc_diff, codes, scale_np

pytestmark = pytest.mark.gpu

SWEEP_NK = [(4096, 7168), (7168, 18432), (18432, 7168), (24576, 1536), (32768, 512),
            (7168, 16384)]
SMALL_M = [1, 8, 16, 40, 64, 65, 128]


@pytest.mark.slow
@pytest.mark.parametrize("N,K", SWEEP_NK)
def test_small_m_sweep_weights(cuda_lib, orc, N, K):
    """m in {1, 8, 16, 40, 64, 65, 128} against each of the six sweep weights at
    full size, quant -> GEMM as the bench runs it: quant codes and scales of
    the checked rows bit-exact, GEMM rows (all rows for m <= 16, else first,
    last and two seeded rows) within tolerance in every column."""
    bfq = cuda_lib
    w = synth.weight(N, K, seed=N + K + 3)
    owq, osw = orc.weight_block_quant(bits(w), False)
    wn = np.linalg.norm(orc.dequant_weight(owq, osw), axis=1)
    d_wq = torch.from_numpy(owq).cuda().view(torch.float8_e4m3fn)
    d_sw = torch.from_numpy(osw).cuda()
    del w
    for M in SMALL_M:
        x = synth.activation(M, K, seed=M * 17 + N + K, zero_group=True)
        q, s = bfq.quant(x.cuda(), 0)
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        bfq.gemm(q, s, 0, d_wq, d_sw, out=out)
        torch.cuda.synchronize()
        rng = np.random.default_rng(M + N + K)
        rows = np.arange(M) if M <= 16 else np.unique(
            np.concatenate([[0, M - 1], rng.integers(0, M, 2)]))
        oq, osa = orc.quant(bits(x[torch.from_numpy(rows)]), 0)
        assert np.array_equal(codes(q)[rows], oq)
        assert np.array_equal(scale_np(s, 0)[:, rows], osa[:, :len(rows)])
        ref = orc.gemm(oq, osa, 0, owq, osw)
        an = np.linalg.norm(orc.dequant_rows(oq, osa, 0), axis=1)
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all(), f"m={M}: rows not written"
        assert_gemm_close(got[rows], ref, an, wn, f"small m={M} n={N} k={K}")
        assert calc_diff(got[rows], ref) < 1e-4


def _problem(orc, M, N, K, fmt, seed):
    x = synth.activation(M, K, seed=seed, zero_group=M * K >= 4096)
    w = synth.weight(N, K, seed=seed + 1)
    aq, sa = orc.quant(bits(x), fmt)
    wq, sw = orc.weight_block_quant(bits(w), fmt != 0)
    dev = (torch.from_numpy(aq).cuda().view(torch.float8_e4m3fn),
           torch.from_numpy(sa.view(np.int32) if fmt == 2 else sa).cuda(),
           torch.from_numpy(wq).cuda().view(torch.float8_e4m3fn),
           torch.from_numpy(sw).cuda())
    return aq, sa, wq, sw, dev


# (M, N, K): ragged row counts from 1 to 127; a last output tile half full
# (N % 256 == 64 or 192); a single K block; K split 2..8 ways over a cluster;
# more tiles than SMs (the persistent walk); one tile with a long K.
EDGES = [(1, 64, 128), (3, 192, 256), (17, 4160, 640), (33, 1088, 1024), (64, 64, 128),
         (64, 19968, 384), (5, 38912, 256), (64, 1024, 18432), (16, 128, 2048),
         (48, 2432, 3200), (65, 320, 4096), (100, 64, 128), (127, 320, 4096)]


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", EDGES)
def test_small_m_edges(cuda_lib, orc, fmt, M, N, K):
    """Every scale format against the oracle; repeated calls bit-identical."""
    bfq = cuda_lib
    aq, sa, wq, sw, d = _problem(orc, M, N, K, fmt, seed=3 * M + N + K + fmt)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm(d[0], d[1], fmt, d[2], d[3], out=out)
    again = bfq.gemm(d[0], d[1], fmt, d[2], d[3])
    torch.cuda.synchronize()
    assert torch.equal(out, again), "repeated calls differ"
    ref = orc.gemm(aq, sa, fmt, wq, sw)
    an = np.linalg.norm(orc.dequant_rows(aq, sa, fmt), axis=1)
    wn = np.linalg.norm(orc.dequant_weight(wq, sw), axis=1)
    assert_gemm_close(out.float().cpu().numpy(), ref, an, wn, f"edge {M}x{N}x{K} fmt{fmt}")


def test_small_m_output_rows_only(cuda_lib, orc):
    """The output buffer is exactly [M][N]: a guard band after it (a larger
    allocation viewed as [M][N]) is never written."""
    bfq = cuda_lib
    M, N, K = 9, 2048, 1024
    aq, sa, wq, sw, d = _problem(orc, M, N, K, 0, seed=71)
    buf = torch.full(((M + 7) * N,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[:M * N].view(M, N)
    bfq.gemm(d[0], d[1], 0, d[2], d[3], out=out)
    torch.cuda.synchronize()
    assert torch.isnan(buf[M * N:]).all(), "wrote past the output"
    ref = orc.gemm(aq, sa, 0, wq, sw)
    an = np.linalg.norm(orc.dequant_rows(aq, sa, 0), axis=1)
    wn = np.linalg.norm(orc.dequant_weight(wq, sw), axis=1)
    assert_gemm_close(out.float().cpu().numpy(), ref, an, wn, "guarded")
