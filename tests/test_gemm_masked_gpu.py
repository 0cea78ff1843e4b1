"""Masked grouped block-scaled FP8 GEMM on the GPU vs the oracle ("[Kernel]
Integrate batched/masked deepgemm kernel"): valid rows within tolerance,
rows r >= count never written, NaN codes in padded rows never spread."""
import numpy as np
import pytest
import torch

import bfq_synth as synth
from helpers import assert_gemm_close, bits, codes

pytestmark = pytest.mark.gpu


def _expert_problem(orc, E, T, N, K, counts, fmt, seed, experts=None):
    """Oracle-quantized per-expert operands; padded activation rows hold the
    e4m3 NaN code 0x7F so any read of them would poison the result."""
    x = synth.masked_activation(E, T, K, torch.from_numpy(counts), seed=seed, poison=False)
    w = synth.expert_weights(E, N, K, seed=seed + 1)
    cols = orc.scale_cols(K, fmt)
    ld = orc.align4(T)
    aq = np.full((E, T, K), 0x7F, np.uint8)
    sa = np.zeros((E, cols, ld), np.uint32 if fmt == 2 else np.float32)
    wq = np.zeros((E, N, K), np.uint8)
    sw = np.zeros((E, (N + 127) // 128, K // 128), np.float32)
    for e in range(E):
        q, s = orc.quant(bits(x[e]), fmt)
        c = counts[e]
        aq[e, :c] = q[:c]
        sa[e] = s
        if experts is None or e in experts:
            wq[e], sw[e] = orc.weight_block_quant(bits(w[e]), fmt != 0)
    return aq, sa, wq, sw, w


def _run_and_check(bfq, orc, aq, sa, wq, sw, counts, fmt, experts=None):
    E, T, K = aq.shape
    N = wq.shape[1]
    d_aq = torch.from_numpy(aq).cuda().view(torch.float8_e4m3fn)
    d_sa = torch.from_numpy(sa.view(np.int32) if fmt == 2 else sa).cuda()
    d_wq = torch.from_numpy(wq).cuda().view(torch.float8_e4m3fn)
    d_sw = torch.from_numpy(sw).cuda()
    d_cnt = torch.from_numpy(counts).cuda()
    out = torch.full((E, T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm_masked(d_aq, d_sa, fmt, d_wq, d_sw, d_cnt, out=out)
    torch.cuda.synchronize()
    oh = out.float().cpu().numpy()
    for e in range(E):
        c = max(0, min(int(counts[e]), T))
        assert np.isnan(oh[e, c:]).all(), f"expert {e}: padded rows written"
        if c == 0 or (experts is not None and e not in experts):
            continue
        rows = np.arange(c) if experts is None else np.unique([0, c // 2, c - 1])
        ref = orc.gemm(aq[e, :c], sa[e], fmt, wq[e], sw[e], rows=rows)
        an = np.linalg.norm(orc.dequant_rows(aq[e, rows], sa[e][:, rows], fmt), axis=1)
        wn = np.linalg.norm(orc.dequant_weight(wq[e], sw[e]), axis=1)
        assert_gemm_close(oh[e, rows], ref, an, wn, f"expert {e}")
    return out


@pytest.mark.parametrize("fmt", [0, 2])
@pytest.mark.parametrize("counts", [[0, 136, 70], [1, 128, 129], [136, 0, 0]])
def test_masked_gemm_small(cuda_lib, orc, fmt, counts):
    E, T, N, K = 3, 136, 320, 384
    cnt = np.array(counts, np.int32)
    aq, sa, wq, sw, _ = _expert_problem(orc, E, T, N, K, cnt, fmt, seed=sum(counts) + fmt)
    _run_and_check(cuda_lib, orc, aq, sa, wq, sw, cnt, fmt)


def test_masked_equals_dense_per_expert(cuda_lib, orc):
    bfq = cuda_lib
    E, T, N, K = 2, 64, 256, 512
    cnt = np.array([64, 33], np.int32)
    aq, sa, wq, sw, _ = _expert_problem(orc, E, T, N, K, cnt, 2, seed=17)
    out = _run_and_check(bfq, orc, aq, sa, wq, sw, cnt, 2)
    for e in range(E):
        c = int(cnt[e])
        d_aq = torch.from_numpy(aq[e, :c].copy()).cuda().view(torch.float8_e4m3fn)
        d_sa = torch.from_numpy(sa[e].view(np.int32)[:, :].copy()).cuda()
        dense = torch.empty((c, N), dtype=torch.bfloat16, device="cuda")
        bfq.bfq_gemm_block_fp8(d_aq, d_sa, 2, d_sa.shape[-1],
                               torch.from_numpy(wq[e]).cuda().view(torch.float8_e4m3fn),
                               torch.from_numpy(sw[e]).cuda(), dense, None)
        torch.cuda.synchronize()
        assert torch.equal(dense, out[e, :c])


@pytest.mark.slow
@pytest.mark.parametrize("N,K", [(4096, 7168), (7168, 2048)])
def test_masked_moe_config_sampled(cuda_lib, orc, N, K):
    """E = 32, T_max = 256, counts ~ U{0..256}: all experts' padded rows are
    checked, sampled rows of four experts against the oracle."""
    E, T = 32, 256
    cnt = synth.valid_counts(E, T).numpy()
    nz = [e for e in range(E) if cnt[e] > 0]
    experts = {nz[0], nz[len(nz) // 3], nz[2 * len(nz) // 3], nz[-1]}
    aq, sa, wq, sw, _ = _expert_problem(orc, E, T, N, K, cnt, 2, seed=N, experts=experts)
    _run_and_check(cuda_lib, orc, aq, sa, wq, sw, cnt, 2, experts=experts)


def test_moe_expert_slice_chain(cuda_lib, orc):
    """up GEMM -> silu-mul-quant -> down GEMM over masked experts, against the
    oracle chain (the oracle's up result rounded to bf16, as the GPU stores
    it).  Rows past each count stay untouched end to end."""
    bfq = cuda_lib
    E, T, H, I = 3, 136, 512, 256
    cnt = np.array([70, 0, 136], np.int32)
    x = synth.masked_activation(E, T, H, torch.from_numpy(cnt), seed=401, poison=False)
    w_up = synth.expert_weights(E, 2 * I, H, seed=402)
    w_dn = synth.expert_weights(E, H, I, seed=403)
    d_cnt = torch.from_numpy(cnt).cuda()
    # GPU chain
    a_up = torch.zeros((E, T, H), dtype=torch.float8_e4m3fn, device="cuda")
    sa_up = torch.zeros((E, bfq.scale_cols(H, 2), T), dtype=torch.int32, device="cuda")
    for e in range(E):
        if cnt[e]:
            bfq.bfq_quant(x[e, :cnt[e]].cuda(), a_up[e, :cnt[e]], sa_up[e], 2, T)
    wq_up, sw_up = bfq.weight_block_quant(w_up.cuda(), 1)
    wq_dn, sw_dn = bfq.weight_block_quant(w_dn.cuda(), 1)
    h = torch.full((E, T, 2 * I), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm_masked(a_up, sa_up, 2, wq_up, sw_up, d_cnt, out=h)
    a_dn, sa_dn = bfq.silu_mul_quant(h, d_cnt, 2)
    out = torch.full((E, T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm_masked(a_dn, sa_dn, 2, wq_dn, sw_dn, d_cnt, out=out)
    torch.cuda.synchronize()
    oh = out.float().cpu().numpy()
    # oracle chain
    for e in range(E):
        c = int(cnt[e])
        assert np.isnan(oh[e, c:]).all()
        if c == 0:
            continue
        oq, osa = orc.quant(bits(x[e, :c]), 2, scale_ld=T)
        owq, osw = orc.weight_block_quant(bits(w_up[e]), True)
        up = orc.gemm(oq, osa, 2, owq, osw)                       # fp64 [c, 2I]
        h_bits = bits(torch.from_numpy(up).to(torch.bfloat16))     # bf16 RNE, as stored
        hq, hs = orc.silu_mul_quant(h_bits.reshape(1, c, 2 * I), np.array([c], np.int32), 2,
                                    scale_ld=T)
        dq, dsw = orc.weight_block_quant(bits(w_dn[e]), True)
        ref = orc.gemm(hq[0], hs[0], 2, dq, dsw)
        an = np.linalg.norm(orc.dequant_rows(hq[0], hs[0], 2), axis=1)
        wn = np.linalg.norm(orc.dequant_weight(dq, dsw), axis=1)
        err = np.abs(oh[e, :c] - ref) / (an[:, None] * wn[None, :])
        assert np.isfinite(oh[e, :c]).all() and err.max() <= 2e-3, (e, float(err.max()))


def test_masked_gemm_more_tiles_than_sms(cuda_lib, orc):
    """16 experts with counts from 0 to 256 over 10 column tiles: 210 valid
    tiles, more than one per SM, so the persistent schedule walks several
    per CTA.  Every expert's padded rows stay untouched; first, middle and
    last valid rows of every non-empty expert match the oracle."""
    E, T, N, K = 16, 256, 2560, 256
    cnt = np.array([0, 1, 127, 128, 129, 256, 255, 64, 200, 0, 17, 256, 130, 90, 3, 240],
                   np.int32)
    experts = {e for e in range(E) if cnt[e] > 0}
    aq, sa, wq, sw, _ = _expert_problem(orc, E, T, N, K, cnt, 2, seed=123, experts=experts)
    _run_and_check(cuda_lib, orc, aq, sa, wq, sw, cnt, 2, experts=experts)


@pytest.mark.parametrize("E,T,N,K,fmt", [(3, 136, 128, 256, 0), (1100, 16, 256, 128, 2)])
def test_masked_gemm_per_tile_forms(cuda_lib, orc, E, T, N, K, fmt):
    """The per-tile masked kernel: 128-wide tiles (N <= 128), and more experts
    than the persistent schedule's prefix table holds (E > 1024).  Padded
    rows of every expert stay untouched; sampled rows of a spread of experts
    match the oracle."""
    rng = np.random.default_rng(E + N)
    cnt = rng.integers(0, T + 1, E).astype(np.int32)
    cnt[0], cnt[-1] = 0, T
    nz = [e for e in range(E) if cnt[e] > 0]
    experts = set(nz[:: max(1, len(nz) // 6)]) | {nz[-1]}
    aq, sa, wq, sw, _ = _expert_problem(orc, E, T, N, K, cnt, fmt, seed=E + T, experts=experts)
    _run_and_check(cuda_lib, orc, aq, sa, wq, sw, cnt, fmt, experts=experts)
