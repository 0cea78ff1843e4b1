"""Masked up projection with silu-and-mul and its quant fused into the GEMM
epilogue (bfq_gemm_block_fp8_masked_silu_quant): the e4m3 codes and scales
must equal, bit for bit, the unfused chain — masked GEMM to a bf16 [E, T, 2I]
output, then bfq_silu_mul_quant — and the oracle's silu-mul-quant of that
bf16 output; rows past each expert's count are never written.  ("[EP+DP]
Optimize the little operations in the DeepGEMM + DeepEP low latency case",
Summary item 2; "[Kernel] Integrate batched/masked deepgemm kernel".)"""
import numpy as np
import pytest
import torch

import bfq_synth as synth
from helpers import bits, codes, scale_np

pytestmark = pytest.mark.gpu

SENT = 0x3C3C3C3C


def test_interleave_gate_up_is_the_block_permutation(cuda_lib):
    bfq = cuda_lib
    E, I, K = 2, 384, 256
    w = torch.randint(0, 256, (E, 2 * I, K), dtype=torch.uint8)
    sw = torch.rand(E, 2 * I // 128, K // 128)
    wo, so = bfq.interleave_gate_up(w.cuda(), sw.cuda())
    torch.cuda.synchronize()
    G = I // 128
    order = [j if b % 2 == 0 else G + j for j in range(G) for b in (0, 1)]
    want_w = w.view(E, 2 * G, 128, K)[:, order].reshape(E, 2 * I, K)
    want_s = sw[:, order]
    assert torch.equal(wo.cpu(), want_w)
    assert torch.equal(so.cpu(), want_s)


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("E,T,H,I,counts", [
    (3, 136, 512, 256, [70, 0, 136]),
    (4, 256, 384, 384, [1, 128, 129, 256]),   # G = 3: a packed word left partial
])
def test_fused_silu_quant_equals_unfused_chain(cuda_lib, orc, fmt, E, T, H, I, counts):
    bfq = cuda_lib
    cnt = np.array(counts, np.int32)
    d_cnt = torch.from_numpy(cnt).cuda()
    a_fmt = 2 if fmt == 2 else 0
    x = synth.masked_activation(E, T, H, torch.from_numpy(cnt), seed=E * 100 + I, poison=False)
    a = torch.zeros((E, T, H), dtype=torch.float8_e4m3fn, device="cuda")
    sa = torch.zeros((E, bfq.scale_cols(H, a_fmt), T), dtype=bfq.scale_dtype(a_fmt), device="cuda")
    for e in range(E):
        if cnt[e]:
            bfq.bfq_quant(x[e, :cnt[e]].cuda(), a[e, :cnt[e]], sa[e], a_fmt, T)
    w = synth.expert_weights(E, 2 * I, H, seed=E * 100 + I + 1)
    wq, sw = bfq.weight_block_quant(w.cuda(), 1 if fmt == 2 else fmt)
    # unfused: masked GEMM to bf16 h, then the silu-mul-quant kernel
    h = torch.full((E, T, 2 * I), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm_masked(a, sa, a_fmt, wq, sw, d_cnt, out=h)
    q_u, sc_u = bfq.silu_mul_quant(h, d_cnt, fmt)
    # fused
    wq_i, sw_i = bfq.interleave_gate_up(wq, sw)
    q_f = torch.full((E, T, I), 0x7E, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    sc_f = torch.full((E, bfq.scale_cols(I, fmt), T), SENT, dtype=torch.int32, device="cuda")
    bfq.bfq_gemm_block_fp8_masked_silu_quant(a, sa, a_fmt, T, wq_i, sw_i, d_cnt, fmt, q_f, sc_f, T)
    torch.cuda.synchronize()
    qf, qu = codes(q_f), codes(q_u)
    sf, su = scale_np(sc_f, fmt), scale_np(sc_u, fmt)
    sent = np.array([SENT], np.uint32).view(np.float32 if fmt != 2 else np.uint32)[0]
    for e in range(E):
        c = int(cnt[e])
        assert np.array_equal(qf[e, :c], qu[e, :c]), f"expert {e}: codes"
        assert np.array_equal(sf[e][:, :c], su[e][:, :c]), f"expert {e}: scales"
        assert (qf[e, c:] == 0x7E).all(), f"expert {e}: padded rows written"
        assert np.array_equal(sf[e][:, c:], np.full_like(sf[e][:, c:], sent)), \
            f"expert {e}: padded scale columns written"
        if c:
            oq, osc = orc.silu_mul_quant(bits(h[e:e + 1, :c]), np.array([c], np.int32), fmt,
                                         scale_ld=T)
            assert np.array_equal(qf[e, :c], oq[0]), f"expert {e}: codes vs oracle"
            assert np.array_equal(sf[e][:, :c], osc[0][:, :c]), f"expert {e}: scales vs oracle"


@pytest.mark.slow
def test_fused_silu_quant_moe_config(cuda_lib, orc):
    """The MoE config (E=32, T=256, H=7168, I=2048, counts ~U{0..256}, packed
    UE8M0): fused equals the unfused chain on every valid row, and on sampled
    rows (the first and last four valid rows of three experts) the fused
    codes and scales match the oracle's own chain — its quant of the same
    activations, fp64 up projection rounded to bf16, silu-mul-quant — up to
    the rare code that an ulp of the bf16 up output can move."""
    bfq = cuda_lib
    E, T, H, I = 32, 256, 7168, 2048
    counts = synth.valid_counts(E, T)
    d_cnt = counts.cuda()
    x = synth.masked_activation(E, T, H, counts, seed=900, device="cuda", poison=False)
    live = [e for e in range(E) if int(counts[e]) > 0]
    sample = sorted({live[0], live[len(live) // 2], live[-1]})
    x_rows = {}
    for e in sample:
        c = int(counts[e])
        rows = sorted({0, 1, 2, 3, c - 4, c - 3, c - 2, c - 1} & set(range(c)))
        x_rows[e] = (rows, bits(x[e, torch.tensor(rows, device="cuda")]))
    a = torch.zeros((E, T, H), dtype=torch.float8_e4m3fn, device="cuda")
    sa = torch.zeros((E, bfq.scale_cols(H, 2), T), dtype=torch.int32, device="cuda")
    for e in range(E):
        c = int(counts[e])
        if c:
            bfq.bfq_quant(x[e, :c], a[e, :c], sa[e], 2, T)
    del x
    wq = torch.empty((E, 2 * I, H), dtype=torch.float8_e4m3fn, device="cuda")
    sw = torch.empty((E, 2 * I // 128, H // 128), dtype=torch.float32, device="cuda")
    for e in range(E):
        q1, s1 = bfq.weight_block_quant(synth.weight(2 * I, H, seed=700 + e, device="cuda"), 1)
        wq[e].copy_(q1)
        sw[e].copy_(s1)
    h = bfq.gemm_masked(a, sa, 2, wq, sw, d_cnt)
    q_u, sc_u = bfq.silu_mul_quant(h, d_cnt, 2)
    wq_i, sw_i = bfq.interleave_gate_up(wq, sw)
    q_f, sc_f = bfq.gemm_masked_silu_quant(a, sa, 2, wq_i, sw_i, d_cnt, 2)
    torch.cuda.synchronize()
    qf, qu = codes(q_f), codes(q_u)
    sf, su = scale_np(sc_f, 2), scale_np(sc_u, 2)
    for e in range(E):
        c = int(counts[e])
        assert np.array_equal(qf[e, :c], qu[e, :c]), f"expert {e}"
        assert np.array_equal(sf[e][:, :c], su[e][:, :c]), f"expert {e}"
    # the oracle's chain on the sampled rows
    dec = orc.e4m3_decode_table()
    for e in sample:
        rows, xb = x_rows[e]
        n = len(rows)
        owq, osw = orc.weight_block_quant(bits(synth.weight(2 * I, H, seed=700 + e,
                                                           device="cuda")), True)
        oq, osa = orc.quant(xb, 2)
        up = orc.gemm(oq, osa, 2, owq, osw)                      # fp64 [n, 2I]
        hb = bits(torch.from_numpy(up).to(torch.bfloat16))       # bf16 RNE, as stored
        yq, ys = orc.silu_mul_quant(hb.reshape(1, n, 2 * I), np.array([n], np.int32), 2)
        got_q, got_s = qf[e, rows], sf[e][:, rows]
        ref_q, ref_s = yq[0], ys[0][:, :n]
        assert (got_s == ref_s).mean() >= 0.99, f"expert {e}: scales"
        # codes of the groups whose packed scale word agrees (a group's scale
        # moves only if an ulp of its amax crosses a power of two)
        words_ok = (got_s == ref_s).T                                   # [n, I/512]
        group_ok = np.repeat(words_ok, 512, axis=1)[:, :I]              # [n, I]
        same = (got_q == ref_q) | ~group_ok
        assert same.mean() >= 0.999, f"expert {e}: {int((~same).sum())} codes differ"
        # a differing code is at most one e4m3 step away
        diff = np.abs(dec[got_q[~same]] - dec[ref_q[~same]])
        step = np.maximum(np.abs(dec[ref_q[~same]]) * 2.0 ** -3, 2.0 ** -9)
        assert (diff <= step * 1.0001).all(), f"expert {e}: a code moved by more than one step"
