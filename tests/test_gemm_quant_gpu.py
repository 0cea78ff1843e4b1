"""Dense GEMM with the output quant fused into its epilogue
(bfq_gemm_block_fp8_quant): the e4m3 codes and scales must equal, bit for
bit, the per-token-group quant of the GEMM's own bf16 output — checked
against the oracle's quant of that output and against the unfused chain
(bfq_gemm_block_fp8 then bfq_quant) — and the bf16 output must be within the
GEMM tolerance of the oracle.  ("[Perf] Deepgemm fused layout kernel for
activations", Purpose: no separate quant/layout pass; "vLLM DeepGEMM FP8
Block GEMM 基准测试" §4.1 for the quant.)"""
import numpy as np
import pytest
import torch

import bfq_synth as synth
from helpers import assert_gemm_close, bits, codes, scale_np

pytestmark = pytest.mark.gpu

SENT = 0x5A5A5A5A


def _problem(orc, bfq, M, N, K, a_fmt, seed):
    x = synth.activation(M, K, seed=seed)
    w = synth.weight(N, K, seed=seed + 1)
    aq, sa = orc.quant(bits(x), a_fmt)
    wq, sw = orc.weight_block_quant(bits(w), a_fmt != 0)
    d_aq = torch.from_numpy(aq).cuda().view(torch.float8_e4m3fn)
    d_sa = torch.from_numpy(sa.view(np.int32) if a_fmt == 2 else sa).cuda()
    d_wq = torch.from_numpy(wq).cuda().view(torch.float8_e4m3fn)
    d_sw = torch.from_numpy(sw).cuda()
    return (aq, sa, wq, sw), (d_aq, d_sa, d_wq, d_sw)


def _fused(bfq, d, a_fmt, M, N, q_fmt, ld, with_out=True):
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda") if with_out else None
    q = torch.full((M, N), 0x7E, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    sc = torch.full((bfq.scale_cols(N, q_fmt), ld), SENT, dtype=torch.int32, device="cuda")
    bfq.bfq_gemm_block_fp8_quant(d[0], d[1], a_fmt, d[1].shape[-1], d[2], d[3], out, q_fmt, q, sc,
                                 ld)
    torch.cuda.synchronize()
    return out, q, sc


# (M, N, K): ragged tiles, packed scale words left partial (N/128 = 1, 3,
# 10, 19, 33), 128-wide tiles (N = 128), shapes the plain GEMM splits along
# K (through distributed shared memory), one CTA per 128-wide tile (100 x
# 16384) and per 256-wide tile (1024 x 2560), the persistent schedule (with
# a half-full last column tile at 2048 x 2432, a second round of 64 tiles at
# 1536 x 4608 x 4096, and a ragged last row tile at 2000 x 2560), and the
# two-way split of a partial second wave (1280 x 4224 x 8192).
SHAPES = [(40, 384, 1024), (64, 128, 512), (130, 512, 640), (257, 1280, 384), (24, 512, 4096),
          (100, 16384, 256), (1024, 2560, 512), (2048, 2560, 256), (2048, 2432, 384),
          (1280, 4224, 8192), (1536, 4608, 4096), (2000, 2560, 256)]


@pytest.mark.parametrize("q_fmt", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_fused_output_quant_matches_quant_of_output(cuda_lib, orc, q_fmt, M, N, K):
    bfq = cuda_lib
    a_fmt = 2 if q_fmt == 2 else 0
    (aq, sa, wq, sw), d = _problem(orc, bfq, M, N, K, a_fmt, seed=M + N + K + q_fmt)
    ld = bfq.align4(M) + 4
    out, q, sc = _fused(bfq, d, a_fmt, M, N, q_fmt, ld)
    # the bf16 output: within the GEMM tolerance of the oracle (sampled rows
    # for the large shape)
    rows = np.arange(M) if M <= 300 else np.unique(np.r_[0, M - 1, np.arange(5, M, 97)])
    ref = orc.gemm(aq, sa, a_fmt, wq, sw, rows=rows)
    an = np.linalg.norm(orc.dequant_rows(aq[rows], sa[:, rows], a_fmt), axis=1)
    wn = np.linalg.norm(orc.dequant_weight(wq, sw), axis=1)
    got = out.float().cpu().numpy()
    assert_gemm_close(got[rows], ref, an, wn, f"fused gemm {M}x{N}x{K}")
    # the quant: bit for bit the oracle's quant of that bf16 output
    oq, osc = orc.quant(bits(out.cpu()), q_fmt, scale_ld=ld)
    assert np.array_equal(codes(q), oq)
    got_sc = scale_np(sc, q_fmt)
    assert np.array_equal(got_sc[:, :M], osc[:, :M])
    assert (sc[:, M:].cpu().numpy() == SENT).all(), "scale padding columns written"


@pytest.mark.parametrize("q_fmt", [0, 2])
@pytest.mark.parametrize("M,N,K", [(24, 512, 4096), (130, 1280, 640), (1152, 4096, 384),
                                   (2048, 2560, 256)])
def test_fused_equals_unfused_chain_and_out_is_optional(cuda_lib, orc, q_fmt, M, N, K):
    """Same launch plan as the plain GEMM (split along K for the first two,
    one CTA per tile, persistent): the fused codes, scales and bf16 output
    equal the plain GEMM followed by the quant kernel; without the bf16
    output the codes and scales are unchanged."""
    bfq = cuda_lib
    a_fmt = 0
    _, d = _problem(orc, bfq, M, N, K, a_fmt, seed=7 + M + q_fmt)
    ld = bfq.align4(M)
    out, q, sc = _fused(bfq, d, a_fmt, M, N, q_fmt, ld)
    out_u = bfq.gemm(d[0], d[1], a_fmt, d[2], d[3])
    q_u, sc_u = bfq.quant(out_u, q_fmt)
    torch.cuda.synchronize()
    assert torch.equal(out, out_u)
    assert torch.equal(q.view(torch.uint8), q_u.view(torch.uint8))
    assert np.array_equal(scale_np(sc, q_fmt)[:, :M], scale_np(sc_u, q_fmt)[:, :M])
    _, q2, sc2 = _fused(bfq, d, a_fmt, M, N, q_fmt, ld, with_out=False)
    assert torch.equal(q2.view(torch.uint8), q.view(torch.uint8))
    assert torch.equal(sc2, sc)


def test_fused_quant_rejects_unsupported(cuda_lib):
    bfq = cuda_lib
    lib = bfq.load_library()
    a = torch.zeros((8, 256), dtype=torch.uint8, device="cuda")
    s = torch.zeros((2, 8), dtype=torch.float32, device="cuda")
    w = torch.zeros((192, 256), dtype=torch.uint8, device="cuda")
    sw = torch.zeros((2, 2), dtype=torch.float32, device="cuda")
    q = torch.zeros((8, 192), dtype=torch.uint8, device="cuda")
    qs = torch.zeros((2, 8), dtype=torch.float32, device="cuda")
    # N = 192 is not a multiple of 128: no whole output groups
    st = lib.bfq_gemm_block_fp8_quant(a.data_ptr(), s.data_ptr(), 0, 8, w.data_ptr(),
                                      sw.data_ptr(), 8, 192, 256, None, 0, q.data_ptr(),
                                      qs.data_ptr(), 8, None, 0, None)
    assert bfq.STATUS_NAMES[st] == "BFQ_ERR_UNSUPPORTED_SHAPE"
    # scale leading dimension below M
    st = lib.bfq_gemm_block_fp8_quant(a.data_ptr(), s.data_ptr(), 0, 8, w.data_ptr(),
                                      sw.data_ptr(), 8, 128, 256, None, 0, q.data_ptr(),
                                      qs.data_ptr(), 4, None, 0, None)
    assert bfq.STATUS_NAMES[st] == "BFQ_ERR_INVALID_ARG"
