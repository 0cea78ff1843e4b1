"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one oracle function against a definition restated
independently (brute force), a library routine that implements the same
definition (torch's float8_e4m3fn conversion, numpy fp64 matmul, integer
matmul), a closed form, or values worked out by hand.  The pages the oracle
follows are "vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.1-§4.3, vLLM PR #29546
(Purpose), vLLM PR #19885 (Summary item 2) and vLLM PR #19111 (Summary of
Changes).
"""
import math
import os

import numpy as np
import pytest
import torch

import bfq_synth as synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_e4m3(values_f32: np.ndarray) -> np.ndarray:
    """torch's own fp32 -> float8_e4m3fn conversion (RNE), as codes."""
    t = torch.from_numpy(np.ascontiguousarray(values_f32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_from_f32(a) -> np.ndarray:
    return bits_of(torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16))


# ---------------------------------------------------------------------------
# e4m3 format
# ---------------------------------------------------------------------------
def test_e4m3_decode_matches_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.e4m3_decode_table()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan], got[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def _magnitudes(orc):
    return orc.e4m3_decode_table()[:127]


def test_e4m3_encode_matches_torch_on_midpoints_and_random(orc):
    mags = _magnitudes(orc)
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (mags[:-1] + mags[1:]) / 2)  # exact
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    rng = np.random.default_rng(7)
    rnd = np.concatenate([
        rng.uniform(-448, 448, 20000),
        rng.uniform(-2.0 ** -6, 2.0 ** -6, 5000),   # subnormal region of e4m3
        rng.standard_normal(5000) * 10,
    ]).astype(np.float32)
    vals = np.concatenate([mids, -mids, up, dn, -up, -dn, mags.astype(np.float32), rnd])
    got = orc.e4m3_encode(vals)
    ref = torch_e4m3(vals)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def test_e4m3_encode_brute_force_linear_scan(orc):
    """Nearest code by exhaustive scan, ties to the even code, saturating."""
    mags = _magnitudes(orc)
    rng = np.random.default_rng(11)
    vals = np.concatenate([rng.uniform(-500, 500, 3000),
                           rng.uniform(-0.02, 0.02, 3000)]).astype(np.float32)
    got = orc.e4m3_encode(vals)
    for v, c in zip(vals, got):
        a = abs(float(v))
        d = np.abs(mags - a)
        best = np.nonzero(d == d.min())[0]
        code = int(best[0]) if best.size == 1 else int([b for b in best if b % 2 == 0][0])
        if a > 448:
            code = 126
        code |= 0x80 if np.signbit(v) else 0
        assert int(c) == code, (float(v), int(c), code)


@pytest.mark.parametrize("v,code", [
    (448.0, 0x7E), (-448.0, 0xFE), (464.0, 0x7E), (1e6, 0x7E), (-1e6, 0xFE),
    (float("inf"), 0x7E), (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02),
    (1.0, 0x38), (0.0, 0x00), (-0.0, 0x80), (float("nan"), 0x7F),
    (1.0625, 0x38),  # tie between 1.0 (0x38) and 1.125 (0x39): even code
    (1.1875, 0x3A),  # tie between 1.125 (0x39) and 1.25 (0x3A): even code
])
def test_e4m3_encode_special_cases(orc, v, code):
    assert int(orc.e4m3_encode(np.array([v], np.float32))[0]) == code


# ---------------------------------------------------------------------------
# per-token-group quant (1 x 128)
# ---------------------------------------------------------------------------
def _one_group(values, fmt, orc):
    x = np.zeros((1, 128), np.float32)
    x[0, :len(values)] = values
    return orc.quant(bf16_from_f32(x), fmt)


def test_group_scale_hand_computed(orc):
    # amax 448 -> s = 1 exactly, codes are plain e4m3 of the values
    q, s = _one_group([448.0, -224.0, 1.0, 0.5], orc.FMT_F32, orc)
    assert s[0, 0] == np.float32(1.0)
    assert q[0, :4].tolist() == [0x7E, 0xF6, 0x38, 0x30]
    # amax 450 -> fp32 s = fl32(450/448); ue8m0: ceil to 2.0 (byte 128), 450/2 = 225 -> 224
    q, s = _one_group([450.0, 1.0], orc.FMT_F32, orc)
    assert s[0, 0] == np.float32(450.0) / np.float32(448.0)
    assert q[0, 0] == 0x7E
    q, s = _one_group([450.0, 1.0], orc.FMT_F32_POW2, orc)
    assert s[0, 0] == np.float32(2.0) and q[0, 0] == 0x76 and q[0, 1] == 0x30
    q, s = _one_group([450.0, 1.0], orc.FMT_UE8M0_PACKED, orc)
    assert s[0, 0] == 128
    # amax 224 -> s = 0.5 exactly, byte 126
    q, s = _one_group([224.0, -3.0], orc.FMT_UE8M0_PACKED, orc)
    assert s[0, 0] == 126 and q[0, 0] == 0x7E and q[0, 1] == 0xCC  # -6.0


def test_all_zero_group(orc):
    x = np.zeros((2, 256), np.uint16)
    q, s = orc.quant(x, orc.FMT_F32)
    assert not q.any()
    eps_s = np.float32(1e-10) / np.float32(448.0)
    assert np.all(s[:, :2] == eps_s)
    q, s = orc.quant(x, orc.FMT_UE8M0_PACKED)
    # ceil_pow2(1e-10/448 = 2.23e-13) = 2^-42 -> biased exponent 85 for both groups
    assert s[0, 0] == 85 | (85 << 8)
    q, s = orc.quant(x, orc.FMT_F32_POW2)
    assert s[0, 0] == np.float32(2.0 ** -42)


def test_saturating_outlier_maps_to_448(orc):
    x = synth.activation(64, 1024, seed=3, outlier_frac=0.0)
    xf = x.float()
    xf[5, 300] = 50.0 * 9.0
    xf[9, 700] = -50.0 * 7.0
    xb = bits_of(xf.to(torch.bfloat16))
    for fmt in (orc.FMT_F32, orc.FMT_F32_POW2, orc.FMT_UE8M0_PACKED):
        q, _ = orc.quant(xb, fmt)
        if fmt == orc.FMT_F32:
            assert q[5, 300] == 0x7E and q[9, 700] == 0xFE
        assert np.all((q & 0x7F) <= 0x7E)  # never NaN, never beyond 448


def _torch_group_quant(x_bf16: torch.Tensor, pow2: bool):
    """The group-quant definition written with torch ops (fp32 IEEE)."""
    M, K = x_bf16.shape
    xf = x_bf16.float().view(M, K // 128, 128)
    amax = xf.abs().amax(dim=-1, keepdim=True)
    s = torch.clamp(amax, min=1e-10) / 448.0
    if pow2:
        s = torch.exp2(torch.ceil(torch.log2(s)))
    q = (xf / s).to(torch.float8_e4m3fn).view(torch.uint8).view(M, K)
    return q.numpy(), s.view(M, K // 128).numpy()


@pytest.mark.parametrize("pow2", [False, True])
def test_quant_matches_torch_definition(orc, pow2):
    x = synth.activation(37, 1024, seed=5, zero_group=True)
    fmt = orc.FMT_F32_POW2 if pow2 else orc.FMT_F32
    q, s = orc.quant(bits_of(x), fmt)
    qt, st = _torch_group_quant(x, pow2)
    assert np.array_equal(q, qt)
    assert np.array_equal(s[:, :37].T, st)


def test_quant_error_bound(orc):
    x = synth.activation(16, 2048, seed=9)
    q, s = orc.quant(bits_of(x), orc.FMT_F32)
    deq = orc.dequant_rows(q, s, orc.FMT_F32)
    xf = x.double().numpy()
    srep = np.repeat(s[:, :16].T.astype(np.float64), 128, axis=1)
    assert np.all(np.abs(deq - xf) <= 2.0 ** -4 * np.abs(xf) + 2.0 ** -10 * srep)


def _read_packed_golden():
    rows = {}
    with open(os.path.join(GOLDEN, "packed_ue8m0_8x512.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                r, word = line.split()
                rows[int(r)] = int(word, 16)
    return rows


def test_packed_scales_hand_built_example(orc):
    """8 x 512 rows whose group amax is 448 * 2^j, j = ((r + g) mod 5) - 2."""
    M, K = 8, 512
    x = np.zeros((M, K), np.float32)
    for r in range(M):
        for g in range(4):
            j = ((r + g) % 5) - 2
            x[r, g * 128] = 448.0 * 2.0 ** j
            x[r, g * 128 + 1] = -1.0 * 2.0 ** j
    q, s = orc.quant(bf16_from_f32(x), orc.FMT_UE8M0_PACKED)
    expected = _read_packed_golden()
    assert s.shape == (1, 8)
    for r in range(M):
        assert int(s[0, r]) == expected[r], (r, hex(int(s[0, r])))
    # unpacking gives back 2^j; the dequantized values are exact
    deq = orc.dequant_rows(q, s, orc.FMT_UE8M0_PACKED)
    assert np.array_equal(deq, x.astype(np.float64))
    # column-major, TMA-aligned: M = 6 uses ld = 8 and leaves rows 6, 7 untouched
    sent = np.full((1, 8), 0xDEADBEEF, np.uint32)
    q6, s6 = orc.quant(bf16_from_f32(x[:6]), orc.FMT_UE8M0_PACKED, scales_init=sent)
    assert [int(v) for v in s6[0, :6]] == [expected[r] for r in range(6)]
    assert int(s6[0, 6]) == 0xDEADBEEF and int(s6[0, 7]) == 0xDEADBEEF


def test_packed_partial_last_word(orc):
    """K/128 = 6 groups: the second word holds groups 4, 5 and zero bytes."""
    x = np.zeros((1, 768), np.float32)
    for g in range(6):
        x[0, g * 128] = 448.0 * 2.0 ** g
    q, s = orc.quant(bf16_from_f32(x), orc.FMT_UE8M0_PACKED)
    assert s.shape == (2, 4)
    assert int(s[0, 0]) == 127 | 128 << 8 | 129 << 16 | 130 << 24
    assert int(s[1, 0]) == 131 | 132 << 8


# ---------------------------------------------------------------------------
# bfq-exp and silu
# ---------------------------------------------------------------------------
def _ulp_dist(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ia = a.view(np.int32).astype(np.int64)
    ib = b.view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


def test_exp_within_2ulp_of_fp64(orc):
    xs = np.linspace(-87.3, 88.7, 60001).astype(np.float32)
    got = orc.expf(xs)
    ref = np.exp(xs.astype(np.float64)).astype(np.float32)
    assert _ulp_dist(got, ref).max() <= 2


def test_exp_special_values(orc):
    v = orc.expf(np.array([0.0, -88.5, 89.5, -1000, 1000, float("nan")], np.float32))
    assert v[0] == 1.0 and v[1] == 0.0 and v[2] == np.inf and v[3] == 0.0
    assert v[4] == np.inf and np.isnan(v[5])
    xs = np.linspace(-20, 20, 20001).astype(np.float32)
    e = orc.expf(xs)
    assert np.all(np.diff(e.astype(np.float64)) >= 0)  # monotone


def test_silu_against_fp64(orc):
    xs = np.linspace(-30, 30, 30001).astype(np.float32)
    got = orc.silu(xs)
    x64 = xs.astype(np.float64)
    ref = (x64 / (1.0 + np.exp(-x64))).astype(np.float32)
    assert _ulp_dist(got, ref).max() <= 4
    big = orc.silu(np.array([0.0, 100.0, 250.0, -100.0, -250.0], np.float32))
    assert big[0] == 0.0 and big[1] == 100.0 and big[2] == 250.0
    assert abs(big[3]) < 1e-30 and abs(big[4]) < 1e-30


# ---------------------------------------------------------------------------
# fused silu-mul-quant over a masked batch
# ---------------------------------------------------------------------------
def test_silu_mul_quant_against_torch_and_masking(orc):
    E, T, I = 4, 40, 512
    counts = np.array([0, 17, 40, 33], np.int32)
    x = synth.masked_activation(E, T, 2 * I, torch.from_numpy(counts), seed=21)
    xb = bits_of(x)
    q_init = np.full((E, T, I), 0xAB, np.uint8)
    s_init = np.full((E, 1, 40), 0xDEADBEEF, np.uint32)
    q, s = orc.silu_mul_quant(xb, counts, orc.FMT_UE8M0_PACKED, q_init=q_init,
                              scales_init=s_init)
    for e in range(E):
        c = counts[e]
        assert np.all(q[e, c:] == 0xAB) and np.all(s[e, :, c:] == 0xDEADBEEF)
        if c == 0:
            continue
        assert np.all((q[e, :c] & 0x7F) != 0x7F)  # the NaN poison never spread
        xf = x[e, :c].float()
        g, u = xf[:, :I], xf[:, I:]
        y = (g / (1.0 + torch.exp(-g))) * u        # torch's own fp32 exp
        amax = y.view(c, I // 128, 128).abs().amax(-1, keepdim=True)
        st = torch.exp2(torch.ceil(torch.log2(torch.clamp(amax, min=1e-10) / 448.0)))
        qt = (y.view(c, I // 128, 128) / st).to(torch.float8_e4m3fn).view(torch.uint8)
        qt = qt.view(c, I).numpy()
        # exp differs by an ulp between libraries: allow a few one-step code flips
        diff = np.abs(q[e, :c].astype(np.int16) - qt.astype(np.int16))
        assert diff.max() <= 1 and (diff > 0).mean() < 2e-3
        bytes_t = (torch.log2(st).view(c, I // 128).numpy() + 127).astype(np.int64)
        words = s[e, :, :c].astype(np.int64)
        for gi in range(I // 128):
            got_b = (words[gi // 4] >> (8 * (gi % 4))) & 0xFF
            assert np.array_equal(got_b, bytes_t[:, gi])


# ---------------------------------------------------------------------------
# 128 x 128 weight block quant
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("pow2", [False, True])
def test_weight_block_quant_matches_torch(orc, pow2):
    N, K = 320, 384  # a partial last row-block (64 rows)
    w = synth.weight(N, K, seed=13)
    wq, sw = orc.weight_block_quant(bits_of(w), pow2)
    wf = torch.zeros(384, K)
    wf[:N] = w.float()
    blocks = wf.view(3, 128, 3, 128).abs().amax(dim=(1, 3))
    st = torch.clamp(blocks, min=1e-10) / 448.0
    if pow2:
        st = torch.exp2(torch.ceil(torch.log2(st)))
    assert np.array_equal(sw, st.numpy())
    srep = st.repeat_interleave(128, 0).repeat_interleave(128, 1)[:N]
    qt = (w.float() / srep).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(wq, qt)


# ---------------------------------------------------------------------------
# block-scaled GEMM
# ---------------------------------------------------------------------------
def _quantized_problem(orc, M, N, K, fmt, seed):
    x = synth.activation(M, K, seed=seed)
    w = synth.weight(N, K, seed=seed + 1)
    aq, sa = orc.quant(bits_of(x), fmt)
    wq, sw = orc.weight_block_quant(bits_of(w), fmt != orc.FMT_F32)
    return aq, sa, wq, sw


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_gemm_equals_dequantized_fp64_matmul(orc, fmt):
    M, N, K = 7, 200, 640
    aq, sa, wq, sw = _quantized_problem(orc, M, N, K, fmt, seed=31)
    c = orc.gemm(aq, sa, fmt, wq, sw)
    ahat = orc.dequant_rows(aq, sa, fmt)
    what = orc.dequant_weight(wq, sw)
    ref = ahat @ what.T
    norm = np.linalg.norm(ahat, axis=1)[:, None] * np.linalg.norm(what, axis=1)[None, :]
    assert np.max(np.abs(c - ref) / norm) < 1e-13
    if fmt != orc.FMT_F32:  # power-of-two scales: both sums are exact up to ordering
        assert np.max(np.abs(c - ref) / norm) < 1e-15


def test_gemm_small_integers_equal_integer_matmul(orc):
    """Unit scales and small integer codes: the block GEMM is an integer matmul."""
    M, N, K = 5, 9, 256
    rng = np.random.default_rng(4)
    ai = rng.integers(-4, 5, (M, K))
    wi = rng.integers(-4, 5, (N, K))
    int_code = {v: c for c, v in enumerate(orc.e4m3_decode_table()[:127]) if float(v).is_integer()}
    enc = lambda a: np.vectorize(lambda v: int_code[abs(v)] | (0x80 if v < 0 else 0))(a)
    aq, wq = enc(ai).astype(np.uint8), enc(wi).astype(np.uint8)
    sa = np.ones((2, 8), np.float32)
    sw = np.ones((1, 2), np.float32)
    c = orc.gemm(aq, sa, orc.FMT_F32, wq, sw)
    assert np.array_equal(c, (ai @ wi.T).astype(np.float64))


def test_gemm_single_block_isolates_scale_pair(orc):
    M, N, K = 3, 260, 512
    aq, sa, wq, sw = _quantized_problem(orc, M, N, K, orc.FMT_F32, seed=41)
    aq = aq.copy()
    wq = wq.copy()
    keep = slice(256, 384)  # only K-block 2 is non-zero
    mask = np.zeros(K, bool)
    mask[keep] = True
    aq[:, ~mask] = 0
    wq[:, ~mask] = 0
    c = orc.gemm(aq, sa, orc.FMT_F32, wq, sw)
    dec = orc.e4m3_decode_table()
    dots = dec[aq[:, keep]] @ dec[wq[:, keep]].T
    scale = sa[2, :M].astype(np.float64)[:, None] * sw[np.arange(N) // 128, 2].astype(
        np.float64)[None, :]
    assert np.array_equal(c, dots * scale)


def test_gemm_packed_equals_pow2_format(orc):
    M, N, K = 6, 128, 1024
    x = synth.activation(M, K, seed=51)
    w = synth.weight(N, K, seed=52)
    wq, sw = orc.weight_block_quant(bits_of(w), True)
    aq1, sa1 = orc.quant(bits_of(x), orc.FMT_F32_POW2)
    aq2, sa2 = orc.quant(bits_of(x), orc.FMT_UE8M0_PACKED)
    assert np.array_equal(aq1, aq2)
    c1 = orc.gemm(aq1, sa1, orc.FMT_F32_POW2, wq, sw)
    c2 = orc.gemm(aq2, sa2, orc.FMT_UE8M0_PACKED, wq, sw)
    assert np.array_equal(c1, c2)


def test_gemm_row_subset_and_orientation(orc):
    M, N, K = 11, 140, 384
    aq, sa, wq, sw = _quantized_problem(orc, M, N, K, orc.FMT_F32, seed=61)
    full = orc.gemm(aq, sa, orc.FMT_F32, wq, sw)
    assert full.shape == (M, N)
    sub = orc.gemm(aq, sa, orc.FMT_F32, wq, sw, rows=[10, 0, 4])
    assert np.array_equal(sub, full[[10, 0, 4]])
    ahat = orc.dequant_rows(aq, sa, orc.FMT_F32)
    what = orc.dequant_weight(wq, sw)
    # element (m, n) is row m of A against row n of W (not the transpose)
    assert abs(full[3, 77] - float(ahat[3] @ what[77])) < 1e-9 * (
        np.linalg.norm(ahat[3]) * np.linalg.norm(what[77]))


def test_gemm_masked_pins(orc):
    E, T, N, K = 3, 20, 128, 256
    counts = np.array([0, 20, 7], np.int32)
    x = synth.masked_activation(E, T, K, torch.from_numpy(counts), seed=71, poison=False)
    w = synth.expert_weights(E, N, K, seed=72)
    fmt = orc.FMT_UE8M0_PACKED
    aq = np.zeros((E, T, K), np.uint8)
    sa = np.zeros((E, 1, 20), np.uint32)
    wq = np.zeros((E, N, K), np.uint8)
    sw = np.zeros((E, 1, 2), np.float32)
    for e in range(E):
        aq[e], sa[e] = orc.quant(bits_of(x[e]), fmt)
        wq[e], sw[e] = orc.weight_block_quant(bits_of(w[e]), True)
    out = orc.gemm_masked(aq, sa, fmt, wq, sw, counts)
    assert np.all(np.isnan(out[0]))                       # count 0 writes nothing
    assert np.all(np.isnan(out[2, 7:])) and not np.isnan(out[2, :7]).any()
    for e in (1, 2):
        dense = orc.gemm(aq[e], sa[e], fmt, wq[e], sw[e])
        c = counts[e]
        assert np.array_equal(out[e, :c], dense[:c])       # equals the dense call


# ---------------------------------------------------------------------------
# the pages' benchmark formulas, against the numbers the pages print
# ---------------------------------------------------------------------------
def test_metric_formulas_reproduce_printed_table():
    import bench

    path = os.path.join(GOLDEN, "dg_bench_h100_table.txt")
    n = 0
    with open(path) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            m, nn, k, us, tflops, gbs = line.split()
            m, nn, k = int(m), int(nn), int(k)
            us, tflops, gbs = float(us), float(tflops), float(gbs)
            # the time is printed to 0.1 us, i.e. up to 7.3e-4 relative
            assert abs(bench.pages_tflops(m, nn, k, us) - tflops) <= 0.051 + 1e-3 * tflops
            assert abs(bench.pages_gbps(m, nn, k, us) - gbs) <= 0.051 + 1e-3 * gbs
            n += 1
    assert n >= 10
