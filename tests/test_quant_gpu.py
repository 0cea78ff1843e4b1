"""Per-token-group quant (1 x 128) on the GPU vs the CPU oracle: codes and
scales must match bit for bit ("vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.1;
"[Perf] Deepgemm fused layout kernel for activations", Purpose)."""
import numpy as np
import pytest
import torch

import bfq_synth as synth
from helpers import bits, codes, scale_np

pytestmark = pytest.mark.gpu

FMTS = [0, 1, 2]
SENT_F = np.float32(-12345.0)
SENT_U = np.uint32(0xDEADBEEF)


def _run(bfq, x_dev, fmt, ld):
    M, K = x_dev.shape
    q = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=x_dev.device)
    sc = torch.empty((bfq.scale_cols(K, fmt), ld), dtype=bfq.scale_dtype(fmt),
                     device=x_dev.device)
    sent = int(SENT_U.view(np.int32)) if fmt == 2 else float(SENT_F)
    sc.fill_(sent)
    bfq.bfq_quant(x_dev, q, sc, fmt, ld)
    torch.cuda.synchronize()
    return q, sc


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,K", [(1, 128), (3, 640), (37, 1024), (130, 7168), (64, 768),
                                 (257, 512)])
def test_quant_bit_exact_small(cuda_lib, orc, fmt, M, K):
    bfq = cuda_lib
    x = synth.activation(M, K, seed=1000 + M + K, zero_group=True)
    ld = bfq.align4(M) + 4  # padding rows beyond M must stay untouched
    q, sc = _run(bfq, x.cuda(), fmt, ld)
    oq, osc = orc.quant(bits(x), fmt, scale_ld=ld)
    assert np.array_equal(codes(q), oq)
    got = scale_np(sc, fmt)
    assert np.array_equal(got[:, :M], osc[:, :M])
    pad = got[:, M:]
    assert np.all(pad == (SENT_U if fmt == 2 else SENT_F))


def test_quant_row_stride(cuda_lib, orc):
    bfq = cuda_lib
    wide = synth.activation(50, 2048, seed=77)
    x = wide[:, 256:1280]  # K = 1024 with ld_x = 2048
    q, sc = _run(bfq, wide.cuda()[:, 256:1280], 2, 52)
    oq, osc = orc.quant(bits(x.contiguous()), 2, scale_ld=52)
    assert np.array_equal(codes(q), oq)
    assert np.array_equal(scale_np(sc, 2)[:, :50], osc[:, :50])


def test_quant_special_values(cuda_lib, orc):
    """Outliers at +-50x, exact powers of two, ties and tiny values."""
    bfq = cuda_lib
    x = torch.zeros(6, 512)
    x[0, :128] = torch.linspace(-448, 448, 128)
    x[1, 0] = 1e-30
    x[1, 1] = -1e-30
    x[1, 2] = -0.0
    x[2, :] = 3.0
    x[3, 5] = 50 * 4.0
    x[3, 6] = -2.0
    x[4, :] = torch.arange(512) * 2.0 ** -12
    x[5, :128] = -1.0
    xb = x.to(torch.bfloat16)
    for fmt in FMTS:
        q, sc = _run(bfq, xb.cuda(), fmt, 8)
        oq, osc = orc.quant(bits(xb), fmt, scale_ld=8)
        assert np.array_equal(codes(q), oq), fmt
        assert np.array_equal(scale_np(sc, fmt)[:, :6], osc[:, :6]), fmt


def test_quant_empty(cuda_lib):
    bfq = cuda_lib
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((0, 256), dtype=torch.float8_e4m3fn, device="cuda")
    sc = torch.empty((2, 0), dtype=torch.float32, device="cuda")
    bfq.bfq_quant(x, q, sc, 0, 0)


@pytest.mark.parametrize("K", [7168, 18432])
@pytest.mark.parametrize("M", [8, 128, 4096, 16384])
def test_quant_full_size_sampled(cuda_lib, orc, M, K):
    """The standalone-quant workload at full size; the oracle checks sampled
    rows (every row of M <= 128), including the row with the all-zero group."""
    bfq = cuda_lib
    x = synth.activation(M, K, seed=4242 + M, zero_group=True)
    xd = x.cuda()
    zero_rows = torch.nonzero(xd.view(M, K // 128, 128).abs().amax(-1).eq(0).any(-1)).view(-1)
    for fmt in (0, 2):
        q, sc = _run(bfq, xd, fmt, bfq.align4(M))
        if M <= 128:
            rows = np.arange(M)
        else:
            rng = np.random.default_rng(M + K + fmt)
            rows = np.unique(np.concatenate([[0, M - 1], zero_rows.cpu().numpy(),
                                             rng.integers(0, M, 40)]))
        xs = x[torch.from_numpy(rows)]
        oq, osc = orc.quant(bits(xs), fmt)
        assert np.array_equal(codes(q)[rows], oq)
        got = scale_np(sc, fmt)[:, rows]
        assert np.array_equal(got, osc[:, :len(rows)])
        # every code is finite e4m3 (no NaN pattern)
        assert not ((q.view(torch.uint8) & 0x7F) == 0x7F).any().item()
