"""Chains of the hot path captured in CUDA graphs and replayed over fresh
inputs ("vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.2: the wrapper turns on
programmatic dependent launch; "[EP+DP] Optimize the little operations in the
DeepGEMM + DeepEP low latency case", Summary: T_max padding exists so that
the MoE layer can run as a CUDA graph).

Each test captures a chain once, then three times writes new seeded inputs
into the graph's static input buffers (outside the graph), replays it, and
checks the replay against the oracle: quantized codes and scales bit for
bit, GEMM outputs within the 2e-3 gate, padded rows never written.  The
dense chain runs with programmatic dependent launch on and off (the graph
records the launch mode it was captured with)."""
import numpy as np
import pytest
import torch

import bfq_synth as synth
from helpers import assert_gemm_close, bits, codes, scale_np

pytestmark = pytest.mark.gpu


def _capture(fn):
    fn()  # eager run first: per-device set-up happens outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("pdl", [True, False])
def test_graph_quant_gemm_smallest_dense_case(cuda_lib, orc, pdl):
    """quant (1 x 128, fp32 scales) -> GEMM at m=8, n=4096, k=7168."""
    bfq = cuda_lib
    M, N, K = 8, 4096, 7168
    w = synth.weight(N, K, seed=5001)
    owq, osw = orc.weight_block_quant(bits(w), False)
    wn = np.linalg.norm(orc.dequant_weight(owq, osw), axis=1)
    d_wq = torch.from_numpy(owq).cuda().view(torch.float8_e4m3fn)
    d_sw = torch.from_numpy(osw).cuda()
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((M, K), dtype=torch.float8_e4m3fn, device="cuda")
    ld = bfq.align4(M)
    s = torch.empty((K // 128, ld), dtype=torch.float32, device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = bfq.gemm_workspace(M, N, K, x.device)

    def chain():
        bfq.bfq_quant(x, q, s, bfq.SCALE_F32, ld)
        bfq.bfq_gemm_block_fp8(q, s, bfq.SCALE_F32, ld, d_wq, d_sw, out, ws)

    prev = bfq.bfq_set_programmatic_launch(pdl)
    try:
        x.copy_(synth.activation(M, K, seed=5000).cuda())
        g = _capture(chain)
    finally:
        bfq.bfq_set_programmatic_launch(prev)
    for rep in range(3):
        xr = synth.activation(M, K, seed=5010 + rep, zero_group=True)
        x.copy_(xr.cuda())
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        oq, osc = orc.quant(bits(xr), 0, scale_ld=ld)
        assert np.array_equal(codes(q), oq), f"replay {rep}: codes"
        assert np.array_equal(scale_np(s, 0)[:, :M], osc[:, :M]), f"replay {rep}: scales"
        ref = orc.gemm(oq, osc, 0, owq, osw)
        an = np.linalg.norm(orc.dequant_rows(oq, osc, 0), axis=1)
        assert_gemm_close(out.float().cpu().numpy(), ref, an, wn, f"replay {rep}")
    assert bfq.bfq_poll_device_status() == 0


def test_graph_moe_slice_fresh_counts(cuda_lib, orc):
    """Per-expert quant -> masked up GEMM -> silu-mul-quant -> masked down
    GEMM, captured once and replayed with new activations AND new per-expert
    counts (the counts are read on the device, so one graph serves every
    routing); padded rows of the output are never written."""
    bfq = cuda_lib
    E, T, H, I = 3, 136, 512, 256
    fmt = bfq.SCALE_UE8M0_PACKED
    w_up = synth.expert_weights(E, 2 * I, H, seed=5101)
    w_dn = synth.expert_weights(E, H, I, seed=5102)
    up_q = [orc.weight_block_quant(bits(w_up[e]), True) for e in range(E)]
    dn_q = [orc.weight_block_quant(bits(w_dn[e]), True) for e in range(E)]
    d_wup = torch.from_numpy(np.stack([u[0] for u in up_q])).cuda().view(torch.float8_e4m3fn)
    d_sup = torch.from_numpy(np.stack([u[1] for u in up_q])).cuda()
    d_wdn = torch.from_numpy(np.stack([d[0] for d in dn_q])).cuda().view(torch.float8_e4m3fn)
    d_sdn = torch.from_numpy(np.stack([d[1] for d in dn_q])).cuda()
    x = torch.empty((E, T, H), dtype=torch.bfloat16, device="cuda")
    d_cnt = torch.zeros(E, dtype=torch.int32, device="cuda")
    a_up = torch.zeros((E, T, H), dtype=torch.float8_e4m3fn, device="cuda")
    sa_up = torch.zeros((E, bfq.scale_cols(H, fmt), T), dtype=torch.int32, device="cuda")
    h = torch.empty((E, T, 2 * I), dtype=torch.bfloat16, device="cuda")
    a_dn = torch.zeros((E, T, I), dtype=torch.float8_e4m3fn, device="cuda")
    sa_dn = torch.zeros((E, bfq.scale_cols(I, fmt), T), dtype=torch.int32, device="cuda")
    out = torch.empty((E, T, H), dtype=torch.bfloat16, device="cuda")

    def chain():
        for e in range(E):  # every row: padded rows are quantized and never used
            bfq.bfq_quant(x[e], a_up[e], sa_up[e], fmt, T)
        bfq.bfq_gemm_block_fp8_masked(a_up, sa_up, fmt, T, d_wup, d_sup, d_cnt, h)
        bfq.bfq_silu_mul_quant(h, d_cnt, a_dn, sa_dn, fmt, T)
        bfq.bfq_gemm_block_fp8_masked(a_dn, sa_dn, fmt, T, d_wdn, d_sdn, d_cnt, out)

    x.copy_(synth.masked_activation(E, T, H, torch.tensor([T] * E), seed=5100).cuda())
    d_cnt.fill_(T)
    g = _capture(chain)
    for rep, cnt in enumerate(([70, 0, 136], [136, 5, 0], [1, 128, 129])):
        cnt = np.array(cnt, np.int32)
        xr = synth.masked_activation(E, T, H, torch.from_numpy(cnt), seed=5110 + rep,
                                     poison=False)
        x.copy_(xr.cuda())
        d_cnt.copy_(torch.from_numpy(cnt))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        oh = out.float().cpu().numpy()
        for e in range(E):
            c = int(cnt[e])
            assert np.isnan(oh[e, c:]).all(), f"replay {rep} expert {e}: padded rows written"
            if c == 0:
                continue
            oq, osa = orc.quant(bits(xr[e, :c]), fmt, scale_ld=T)
            up = orc.gemm(oq, osa, fmt, up_q[e][0], up_q[e][1])
            h_bits = bits(torch.from_numpy(up).to(torch.bfloat16))  # bf16 RNE, as stored
            hq, hs = orc.silu_mul_quant(h_bits.reshape(1, c, 2 * I), np.array([c], np.int32),
                                        fmt, scale_ld=T)
            ref = orc.gemm(hq[0], hs[0], fmt, dn_q[e][0], dn_q[e][1])
            an = np.linalg.norm(orc.dequant_rows(hq[0], hs[0], fmt), axis=1)
            wn = np.linalg.norm(orc.dequant_weight(dn_q[e][0], dn_q[e][1]), axis=1)
            # the 2e-3 gate only: the GPU's bf16 up output may differ from the
            # oracle's by an ulp, which can move a silu-mul-quant code by one
            err = np.abs(oh[e, :c] - ref) / (an[:, None] * wn[None, :])
            assert np.isfinite(oh[e, :c]).all() and err.max() <= 2e-3, (rep, e, err.max())
    assert bfq.bfq_poll_device_status() == 0
