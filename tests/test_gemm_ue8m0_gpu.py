"""Block-scaled FP8 GEMM for power-of-two (UE8M0) scales, the scales applied
by the tensor cores' block scaling (tcgen05.mma kind::mxf8f6f4.block_scale),
against the oracle ("vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.1–4.2: the
UE8M0 scale form; "[Kernel] Integrate batched/masked deepgemm kernel": the
masked per-expert form).

The result definition is the GEMM's: a power-of-two scale is exact to apply,
so the only difference from the promotion kernel is the fp32 summation
order, and every element must meet the same gate (2e-3 * ||A_hat[m]|| *
||W_hat[n]|| of the oracle's fp64 result, plus the one-bf16-ulp sanity
bound).  Inputs spread the scale exponents over rows and K blocks, so a
scale applied to the wrong row, column block or K block cannot pass."""
import numpy as np
import pytest
import torch

import bfq_synth as synth
from helpers import assert_gemm_close, bits, calc_diff, codes, scale_np

pytestmark = pytest.mark.gpu

BFQ_ERR_FORMAT = 4


def _spread(x: torch.Tensor) -> torch.Tensor:
    """Rows and 128-column blocks multiplied by distinct powers of two
    (2^-5 .. 2^5 over rows, 2^-3 .. 2^3 over blocks), so neighbouring rows
    and K blocks get different scale exponents."""
    M, K = x.shape
    f = torch.tensor([2.0 ** ((r * 5) % 11 - 5) for r in range(M)]).view(M, 1)
    g = torch.tensor([2.0 ** ((b * 3) % 7 - 3) for b in range(K // 128)])
    return (x.float() * f * g.repeat_interleave(128).view(1, K)).to(torch.bfloat16)


def _dense_problem(orc, M, N, K, fmt, seed):
    x = _spread(synth.activation(M, K, seed=seed, zero_group=M * K >= 4096))
    w = synth.weight(N, K, seed=seed + 1)
    aq, sa = orc.quant(bits(x), fmt)
    wq, sw = orc.weight_block_quant(bits(w), True)
    dev = (torch.from_numpy(aq).cuda().view(torch.float8_e4m3fn),
           torch.from_numpy(sa.view(np.int32) if fmt == 2 else sa).cuda(),
           torch.from_numpy(wq).cuda().view(torch.float8_e4m3fn),
           torch.from_numpy(sw).cuda())
    return aq, sa, wq, sw, dev


def _check_dense(orc, out, aq, sa, wq, sw, fmt, what, rows=None):
    """All rows, or the given sample of rows, within the gate in every column."""
    r = np.arange(aq.shape[0]) if rows is None else np.asarray(rows)
    ref = orc.gemm(aq, sa, fmt, wq, sw, rows=r)
    an = np.linalg.norm(orc.dequant_rows(aq[r], sa[:, r], fmt), axis=1)
    wn = np.linalg.norm(orc.dequant_weight(wq, sw), axis=1)
    got = out.float().cpu().numpy()[r]
    assert_gemm_close(got, ref, an, wn, what)
    return got, ref


def _sample_rows(M, seed):
    """First and last rows of every 128-row tile plus seeded rows."""
    rng = np.random.default_rng(seed)
    tiles = np.arange(0, M, 128)
    return np.unique(np.concatenate([tiles, np.minimum(tiles + 127, M - 1),
                                     rng.integers(0, M, 8)]))


def _on_block_scaled_plan(M, N, K):
    """The entry point runs the block-scaled kernel (not the promotion plan
    it keeps for one row tile, K < 1024 or few tiles)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = -(-M // 128) * -(-N // 256)
    return M > 128 and K >= 1024 and 2 * tiles >= sms


# Block-scaled plan (M, N, K): a partial last group of K blocks (9 = 4+4+1,
# 23 = 4*5+3); ragged rows (the last tile 1, 80 or 20 rows); a half-full last
# column tile (N % 256 == 64 or 192); one tile per SM and several per SM.
BS_PLAN = [(1300, 1856, 1152), (129, 19968, 1024), (1024, 8192, 1024), (2000, 2496, 2944),
           (4096, 2304, 1536)]
# Promotion plan through the same entry point: one row tile, K < 1024, few tiles.
PROMO_PLAN = [(1, 64, 128), (128, 256, 512), (77, 1088, 2944), (256, 512, 640),
              (1024, 8192, 256)]


@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("M,N,K", BS_PLAN)
def test_ue8m0_gemm_parity(cuda_lib, orc, fmt, M, N, K):
    """Packed UE8M0 and fp32 power-of-two activation scales on the
    block-scaled kernel: sampled rows (every tile's first and last) in every
    column; repeated calls bit-identical; every element written; no error
    latched."""
    assert _on_block_scaled_plan(M, N, K)
    bfq = cuda_lib
    aq, sa, wq, sw, d = _dense_problem(orc, M, N, K, fmt, seed=7 * M + N + K + fmt)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm_ue8m0(d[0], d[1], fmt, d[2], d[3], out=out)
    again = bfq.gemm_ue8m0(d[0], d[1], fmt, d[2], d[3])
    torch.cuda.synchronize()
    assert bfq.bfq_poll_device_status() == 0
    assert torch.equal(out, again), "repeated calls differ"
    assert not torch.isnan(out).any(), "output not fully written"
    _check_dense(orc, out, aq, sa, wq, sw, fmt, f"ue8m0 {M}x{N}x{K} fmt{fmt}",
                 rows=_sample_rows(M, M + N + K))


@pytest.mark.parametrize("M,N,K", PROMO_PLAN)
def test_ue8m0_entry_on_promotion_plan(cuda_lib, orc, M, N, K):
    """Shapes the entry point hands to the promotion kernel's plan: same
    result definition, all rows checked."""
    assert not _on_block_scaled_plan(M, N, K)
    bfq = cuda_lib
    aq, sa, wq, sw, d = _dense_problem(orc, M, N, K, 2, seed=3 * M + N + K)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm_ue8m0(d[0], d[1], 2, d[2], d[3], out=out)
    torch.cuda.synchronize()
    assert bfq.bfq_poll_device_status() == 0
    _check_dense(orc, out, aq, sa, wq, sw, 2, f"ue8m0 entry {M}x{N}x{K}")


def test_ue8m0_matches_promotion_kernel(cuda_lib, orc):
    """The same UE8M0 problem through both kernels: both within the gate of
    the oracle on sampled rows, and within one bf16 ulp (plus 1e-4 of the
    norms) of each other everywhere — only the fp32 summation order differs."""
    bfq = cuda_lib
    M, N, K = 1024, 2560, 3072
    assert _on_block_scaled_plan(M, N, K)
    aq, sa, wq, sw, d = _dense_problem(orc, M, N, K, 2, seed=99)
    bs = bfq.gemm_ue8m0(d[0], d[1], 2, d[2], d[3])
    pr = bfq.gemm(d[0], d[1], 2, d[2], d[3])
    torch.cuda.synchronize()
    rows = _sample_rows(M, 99)
    got, ref = _check_dense(orc, bs, aq, sa, wq, sw, 2, "block-scaled", rows=rows)
    _check_dense(orc, pr, aq, sa, wq, sw, 2, "promotion", rows=rows)
    assert calc_diff(got, ref) < 1e-4
    an = np.linalg.norm(orc.dequant_rows(aq, sa, 2), axis=1)
    wn = np.linalg.norm(orc.dequant_weight(wq, sw), axis=1)
    b = bs.float().cpu().numpy()
    p = pr.float().cpu().numpy()
    slack = 2.0 ** -7 * np.abs(p) + 1e-4 * an[:, None] * wn[None, :]
    assert (np.abs(b - p) <= slack).all()


def test_ue8m0_output_rows_only(cuda_lib, orc):
    """A guard band after the [M][N] output is never written (the last row
    tile holds 44 rows, clipped by the output tensor map)."""
    bfq = cuda_lib
    M, N, K = 300, 6656, 1024
    assert _on_block_scaled_plan(M, N, K)
    aq, sa, wq, sw, d = _dense_problem(orc, M, N, K, 2, seed=71)
    buf = torch.full(((M + 7) * N,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[:M * N].view(M, N)
    bfq.gemm_ue8m0(d[0], d[1], 2, d[2], d[3], out=out)
    torch.cuda.synchronize()
    assert torch.isnan(buf[M * N:]).all(), "wrote past the output"
    _check_dense(orc, out, aq, sa, wq, sw, 2, "guarded", rows=_sample_rows(M, 71))


def test_ue8m0_rejects_non_pow2_formats(cuda_lib, orc):
    """fp32 activation scales are refused on the host; a weight scale that
    is not a power of two is caught on the device (BFQ_ERR_FORMAT latched)."""
    bfq = cuda_lib
    M, N, K = 256, 10240, 1024
    assert _on_block_scaled_plan(M, N, K)
    aq, sa, wq, sw, d = _dense_problem(orc, M, N, K, 2, seed=5)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    a32 = torch.ones((K // 128, M), dtype=torch.float32, device="cuda")
    with pytest.raises(bfq.BfqError) as ei:
        bfq.bfq_gemm_block_fp8_ue8m0(d[0], a32, 0, M, d[2], d[3], out)
    assert ei.value.status == BFQ_ERR_FORMAT
    assert bfq.bfq_poll_device_status() == 0
    bad_sw = d[3].clone()
    bad_sw[1, 2] *= 1.5
    bfq.bfq_gemm_block_fp8_ue8m0(d[0], d[1], 2, d[1].shape[-1], d[2], bad_sw, out)
    torch.cuda.synchronize()
    assert bfq.bfq_poll_device_status() == BFQ_ERR_FORMAT
    assert bfq.bfq_poll_device_status() == 0  # the poll cleared it
    bfq.bfq_gemm_block_fp8_ue8m0(d[0], d[1], 2, d[1].shape[-1], d[2], d[3], out)
    torch.cuda.synchronize()
    assert bfq.bfq_poll_device_status() == 0
    _check_dense(orc, out, aq, sa, wq, sw, 2, "after a rejected call", rows=_sample_rows(M, 5))


def test_ue8m0_weight_scales_loaded_either_way(cuda_lib, orc):
    """Weight scales 16-byte aligned with K / 128 a multiple of 4 move by bulk
    copies; at a 4-byte offset the kernel loads them into registers: the
    two give the same output bit for bit.  Packed activation scales off a
    16-byte boundary are refused."""
    bfq = cuda_lib
    M, N, K = 512, 9728, 2048
    assert _on_block_scaled_plan(M, N, K)
    aq, sa, wq, sw, d = _dense_problem(orc, M, N, K, 2, seed=77)
    a_out = bfq.gemm_ue8m0(d[0], d[1], 2, d[2], d[3])
    buf = torch.empty(d[3].numel() + 1, dtype=torch.float32, device="cuda")
    sw_off = buf[1:].view_as(d[3])
    sw_off.copy_(d[3])
    assert sw_off.data_ptr() % 16 == 4
    b_out = torch.empty_like(a_out)
    bfq.bfq_gemm_block_fp8_ue8m0(d[0], d[1], 2, d[1].shape[-1], d[2], sw_off, b_out)
    torch.cuda.synchronize()
    assert bfq.bfq_poll_device_status() == 0
    assert torch.equal(a_out, b_out)
    _check_dense(orc, b_out, aq, sa, wq, sw, 2, "register-loaded weight scales",
                 rows=_sample_rows(M, 77))
    sbuf = torch.empty(d[1].numel() + 1, dtype=torch.int32, device="cuda")
    sa_off = sbuf[1:].view_as(d[1])
    sa_off.copy_(d[1])
    with pytest.raises(bfq.BfqError) as ei:
        bfq.bfq_gemm_block_fp8_ue8m0(d[0], sa_off, 2, d[1].shape[-1], d[2], d[3], b_out)
    assert ei.value.status == 3  # BFQ_ERR_MISALIGNED


def _expert_problem(orc, E, T, N, K, counts, seed, experts=None):
    """Per-expert operands with packed UE8M0 activation scales and
    power-of-two weight scales; padded activation rows hold the e4m3 NaN
    code 0x7F so any read of them into a stored row would poison it."""
    x = synth.masked_activation(E, T, K, torch.from_numpy(counts), seed=seed, poison=False)
    w = synth.expert_weights(E, N, K, seed=seed + 1)
    ld = orc.align4(T)
    aq = np.full((E, T, K), 0x7F, np.uint8)
    sa = np.zeros((E, orc.scale_cols(K, 2), ld), np.uint32)
    wq = np.zeros((E, N, K), np.uint8)
    sw = np.ones((E, (N + 127) // 128, K // 128), np.float32)
    for e in range(E):
        q, s = orc.quant(bits(_spread(x[e])), 2)
        c = counts[e]
        aq[e, :c] = q[:c]
        sa[e] = s
        if experts is None or e in experts:
            wq[e], sw[e] = orc.weight_block_quant(bits(w[e]), True)
    return aq, sa, wq, sw


def _run_masked(bfq, orc, aq, sa, wq, sw, counts, experts=None):
    E, T, K = aq.shape
    N = wq.shape[1]
    d_aq = torch.from_numpy(aq).cuda().view(torch.float8_e4m3fn)
    d_sa = torch.from_numpy(sa.view(np.int32)).cuda()
    d_wq = torch.from_numpy(wq).cuda().view(torch.float8_e4m3fn)
    d_sw = torch.from_numpy(sw).cuda()
    d_cnt = torch.from_numpy(counts).cuda()
    out = torch.full((E, T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm_masked_ue8m0(d_aq, d_sa, 2, d_wq, d_sw, d_cnt, out=out)
    torch.cuda.synchronize()
    assert bfq.bfq_poll_device_status() == 0
    oh = out.float().cpu().numpy()
    for e in range(E):
        c = max(0, min(int(counts[e]), T))
        assert np.isnan(oh[e, c:]).all(), f"expert {e}: padded rows written"
        if c == 0 or (experts is not None and e not in experts):
            continue
        rows = np.arange(c) if experts is None else np.unique([0, c // 2, c - 1])
        ref = orc.gemm(aq[e, :c], sa[e], 2, wq[e], sw[e], rows=rows)
        an = np.linalg.norm(orc.dequant_rows(aq[e, rows], sa[e][:, rows], 2), axis=1)
        wn = np.linalg.norm(orc.dequant_weight(wq[e], sw[e]), axis=1)
        assert_gemm_close(oh[e, rows], ref, an, wn, f"expert {e}")
    return out


@pytest.mark.parametrize("counts", [[0, 136, 70], [1, 128, 129], [136, 0, 0]])
def test_ue8m0_masked_small(cuda_lib, orc, counts):
    E, T, N, K = 3, 136, 320, 640
    cnt = np.array(counts, np.int32)
    aq, sa, wq, sw = _expert_problem(orc, E, T, N, K, cnt, seed=sum(counts) + 3)
    _run_masked(cuda_lib, orc, aq, sa, wq, sw, cnt)


def test_ue8m0_masked_more_tiles_than_sms(cuda_lib, orc):
    """16 experts, counts 0..256, 10 column tiles: 210 valid tiles, several
    per CTA of the persistent walk."""
    E, T, N, K = 16, 256, 2560, 512
    cnt = np.array([0, 1, 127, 128, 129, 256, 255, 64, 200, 0, 17, 256, 130, 90, 3, 240],
                   np.int32)
    experts = {e for e in range(E) if cnt[e] > 0}
    aq, sa, wq, sw = _expert_problem(orc, E, T, N, K, cnt, seed=321, experts=experts)
    _run_masked(cuda_lib, orc, aq, sa, wq, sw, cnt, experts=experts)


def test_ue8m0_masked_equals_dense_per_expert(cuda_lib, orc):
    """Each expert's valid rows of the masked form equal the dense form of
    the same kernel on those rows, bit for bit (sizes for which the dense
    entry point runs the block-scaled kernel)."""
    bfq = cuda_lib
    E, T, N, K = 2, 256, 9728, 1024
    cnt = np.array([136, 200], np.int32)
    aq, sa, wq, sw = _expert_problem(orc, E, T, N, K, cnt, seed=17)
    out = _run_masked(bfq, orc, aq, sa, wq, sw, cnt, experts=set(range(E)))
    for e in range(E):
        c = int(cnt[e])
        assert _on_block_scaled_plan(c, N, K)
        d_sa = torch.from_numpy(sa[e].view(np.int32).copy()).cuda()
        dense = torch.empty((c, N), dtype=torch.bfloat16, device="cuda")
        bfq.bfq_gemm_block_fp8_ue8m0(
            torch.from_numpy(aq[e, :c].copy()).cuda().view(torch.float8_e4m3fn), d_sa, 2,
            d_sa.shape[-1], torch.from_numpy(wq[e]).cuda().view(torch.float8_e4m3fn),
            torch.from_numpy(sw[e]).cuda(), dense)
        torch.cuda.synchronize()
        assert torch.equal(dense, out[e, :c])


@pytest.mark.slow
@pytest.mark.parametrize("N,K", [(4096, 7168), (7168, 2048)])
def test_ue8m0_masked_moe_config_sampled(cuda_lib, orc, N, K):
    """E = 32, T_max = 256, counts ~ U{0..256} (the MoE configuration): every
    expert's padded rows checked, sampled rows of four experts against the
    oracle."""
    E, T = 32, 256
    cnt = synth.valid_counts(E, T).numpy()
    nz = [e for e in range(E) if cnt[e] > 0]
    experts = {nz[0], nz[len(nz) // 3], nz[2 * len(nz) // 3], nz[-1]}
    aq, sa, wq, sw = _expert_problem(orc, E, T, N, K, cnt, seed=N + 1, experts=experts)
    _run_masked(cuda_lib, orc, aq, sa, wq, sw, cnt, experts=experts)


@pytest.mark.slow
@pytest.mark.parametrize("N,K", [(4096, 7168), (7168, 18432), (24576, 1536), (32768, 512)])
def test_ue8m0_full_size_sampled(cuda_lib, orc, N, K):
    """m = 4096 at sweep sizes, quant -> block-scaled GEMM on the GPU: GPU
    pow2 weight quant bit-exact, sampled quant rows bit-exact, sampled GEMM
    rows within tolerance in every column."""
    bfq = cuda_lib
    M = 4096
    w = synth.weight(N, K, seed=N + K + 11)
    owq, osw = orc.weight_block_quant(bits(w), True)
    wq, sw = bfq.weight_block_quant(w.cuda(), 1)
    torch.cuda.synchronize()
    assert np.array_equal(codes(wq), owq) and np.array_equal(sw.cpu().numpy(), osw)
    wn = np.linalg.norm(orc.dequant_weight(owq, osw), axis=1)
    del w
    x = synth.activation(M, K, seed=M + N + K)
    q, s = bfq.quant(x.cuda(), 2)
    out = bfq.gemm_ue8m0(q, s, 2, wq, sw)
    torch.cuda.synchronize()
    assert bfq.bfq_poll_device_status() == 0
    rng = np.random.default_rng(N + K)
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], rng.integers(0, M, 4)]))
    oq, osa = orc.quant(bits(x[torch.from_numpy(rows)]), 2)
    assert np.array_equal(codes(q)[rows], oq)
    assert np.array_equal(scale_np(s, 2)[:, rows], osa[:, :len(rows)])
    ref = orc.gemm(oq, osa, 2, owq, osw)
    an = np.linalg.norm(orc.dequant_rows(oq, osa, 2), axis=1)
    got = out.float().cpu().numpy()[rows]
    assert_gemm_close(got, ref, an, wn, f"ue8m0 m={M} n={N} k={K}")
    assert calc_diff(got, ref) < 1e-4


SENT = 0x3C3C3C3C


@pytest.mark.parametrize("q_fmt", [0, 1, 2])
@pytest.mark.parametrize("E,T,H,I,counts", [
    (3, 136, 512, 256, [70, 0, 136]),
    (4, 256, 1152, 384, [1, 128, 129, 256]),   # 9 K blocks; a packed word left partial
])
def test_ue8m0_fused_silu_quant_equals_unfused_chain(cuda_lib, orc, q_fmt, E, T, H, I, counts):
    """The up projection with silu-mul-quant in the block-scaled kernel's
    epilogue equals, bit for bit, the block-scaled masked GEMM to bf16
    followed by the silu-mul-quant kernel, and the oracle's silu-mul-quant of
    that bf16 output; padded rows and scale columns are never written."""
    bfq = cuda_lib
    cnt = np.array(counts, np.int32)
    d_cnt = torch.from_numpy(cnt).cuda()
    x = synth.masked_activation(E, T, H, torch.from_numpy(cnt), seed=E * 100 + I + 7,
                                poison=False)
    a = torch.zeros((E, T, H), dtype=torch.float8_e4m3fn, device="cuda")
    sa = torch.zeros((E, bfq.scale_cols(H, 2), T), dtype=torch.int32, device="cuda")
    for e in range(E):
        if cnt[e]:
            bfq.bfq_quant(_spread(x[e, :cnt[e]]).cuda(), a[e, :cnt[e]], sa[e], 2, T)
    w = synth.expert_weights(E, 2 * I, H, seed=E * 100 + I + 8)
    wq, sw = bfq.weight_block_quant(w.cuda(), 1)
    h = torch.full((E, T, 2 * I), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm_masked_ue8m0(a, sa, 2, wq, sw, d_cnt, out=h)
    q_u, sc_u = bfq.silu_mul_quant(h, d_cnt, q_fmt)
    wq_i, sw_i = bfq.interleave_gate_up(wq, sw)
    q_f = torch.full((E, T, I), 0x7E, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    sc_f = torch.full((E, bfq.scale_cols(I, q_fmt), T), SENT, dtype=torch.int32, device="cuda")
    bfq.bfq_gemm_block_fp8_masked_silu_quant_ue8m0(a, sa, 2, T, wq_i, sw_i, d_cnt, q_fmt, q_f,
                                                   sc_f, T)
    torch.cuda.synchronize()
    assert bfq.bfq_poll_device_status() == 0
    qf, qu = codes(q_f), codes(q_u)
    sf, su = scale_np(sc_f, q_fmt), scale_np(sc_u, q_fmt)
    sent = np.array([SENT], np.uint32).view(np.float32 if q_fmt != 2 else np.uint32)[0]
    for e in range(E):
        c = int(cnt[e])
        assert np.array_equal(qf[e, :c], qu[e, :c]), f"expert {e}: codes"
        assert np.array_equal(sf[e][:, :c], su[e][:, :c]), f"expert {e}: scales"
        assert (qf[e, c:] == 0x7E).all(), f"expert {e}: padded rows written"
        assert np.array_equal(sf[e][:, c:], np.full_like(sf[e][:, c:], sent)), \
            f"expert {e}: padded scale columns written"
        if c:
            oq, osc = orc.silu_mul_quant(bits(h[e:e + 1, :c]), np.array([c], np.int32), q_fmt,
                                         scale_ld=T)
            assert np.array_equal(qf[e, :c], oq[0]), f"expert {e}: codes vs oracle"
            assert np.array_equal(sf[e][:, :c], osc[0][:, :c]), f"expert {e}: scales vs oracle"


@pytest.mark.slow
def test_ue8m0_fused_silu_quant_moe_config(cuda_lib, orc):
    """The MoE configuration (E=32, T=256, H=7168, I=2048, counts ~U{0..256},
    packed UE8M0): fused equals the unfused block-scaled chain on every valid
    row; on three experts the fused codes and scales equal the oracle's
    silu-mul-quant of the GPU's bf16 up output."""
    bfq = cuda_lib
    E, T, H, I = 32, 256, 7168, 2048
    counts = synth.valid_counts(E, T)
    d_cnt = counts.cuda()
    x = synth.masked_activation(E, T, H, counts, seed=901, device="cuda", poison=False)
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
    h = bfq.gemm_masked_ue8m0(a, sa, 2, wq, sw, d_cnt)
    q_u, sc_u = bfq.silu_mul_quant(h, d_cnt, 2)
    wq_i, sw_i = bfq.interleave_gate_up(wq, sw)
    del wq, sw
    q_f = torch.empty((E, T, I), dtype=torch.float8_e4m3fn, device="cuda")
    sc_f = torch.empty((E, bfq.scale_cols(I, 2), T), dtype=torch.int32, device="cuda")
    bfq.bfq_gemm_block_fp8_masked_silu_quant_ue8m0(a, sa, 2, T, wq_i, sw_i, d_cnt, 2, q_f, sc_f,
                                                   T)
    torch.cuda.synchronize()
    assert bfq.bfq_poll_device_status() == 0
    qf, qu = codes(q_f), codes(q_u)
    sf, su = scale_np(sc_f, 2), scale_np(sc_u, 2)
    live = [e for e in range(E) if int(counts[e]) > 0]
    for e in range(E):
        c = int(counts[e])
        assert np.array_equal(qf[e, :c], qu[e, :c]), f"expert {e}"
        assert np.array_equal(sf[e][:, :c], su[e][:, :c]), f"expert {e}"
    for e in sorted({live[0], live[len(live) // 2], live[-1]}):
        c = int(counts[e])
        oq, osc = orc.silu_mul_quant(bits(h[e:e + 1, :c]), np.array([c], np.int32), 2,
                                     scale_ld=T)
        assert np.array_equal(qf[e, :c], oq[0]) and np.array_equal(sf[e][:, :c], osc[0][:, :c])
