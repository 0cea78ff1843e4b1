"""Dense block-scaled FP8 GEMM on the GPU vs the oracle's fp64 result
("vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.2): every checked element within
2e-3 * ||A_hat[m]|| * ||W_hat[n]||, plus a one-bf16-ulp sanity bound."""
import numpy as np
import pytest
import torch

import bfq_synth as synth
from helpers import assert_gemm_close, bits, calc_diff, codes, scale_np

pytestmark = pytest.mark.gpu


def _oracle_problem(orc, M, N, K, fmt, seed):
    x = synth.activation(M, K, seed=seed, zero_group=M * K >= 4096)
    w = synth.weight(N, K, seed=seed + 1)
    aq, sa = orc.quant(bits(x), fmt)
    wq, sw = orc.weight_block_quant(bits(w), fmt != 0)
    return aq, sa, wq, sw


def _to_dev(aq, sa, wq, sw, fmt):
    d_aq = torch.from_numpy(aq).cuda().view(torch.float8_e4m3fn)
    d_sa = torch.from_numpy(sa.view(np.int32) if fmt == 2 else sa).cuda()
    d_wq = torch.from_numpy(wq).cuda().view(torch.float8_e4m3fn)
    d_sw = torch.from_numpy(sw).cuda()
    return d_aq, d_sa, d_wq, d_sw


def _norms(orc, aq, sa, wq, sw, fmt, rows=None):
    r = slice(None) if rows is None else rows
    an = np.linalg.norm(orc.dequant_rows(aq[r], sa[:, r] if rows is not None else sa, fmt),
                        axis=1)
    wn = np.linalg.norm(orc.dequant_weight(wq, sw), axis=1)
    return an, wn


SMALL = [(1, 64, 128), (8, 256, 1024), (40, 384, 1024), (130, 320, 640), (200, 512, 2048),
         (257, 192, 384), (128, 128, 256), (300, 1024, 512)]


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_gemm_parity_small(cuda_lib, orc, fmt, M, N, K):
    bfq = cuda_lib
    aq, sa, wq, sw = _oracle_problem(orc, M, N, K, fmt, seed=7 * M + N + K + fmt)
    d = _to_dev(aq, sa, wq, sw, fmt)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm(d[0], d[1], fmt, d[2], d[3], out=out)
    torch.cuda.synchronize()
    ref = orc.gemm(aq, sa, fmt, wq, sw)
    an, wn = _norms(orc, aq, sa, wq, sw, fmt)
    assert_gemm_close(out.float().cpu().numpy(), ref, an, wn, f"gemm {M}x{N}x{K} fmt{fmt}")


def _no_workspace_gemm(bfq, d, fmt, out=None):
    """The dense GEMM called with no workspace: the plans that need none."""
    M, N = d[0].shape[0], d[2].shape[0]
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda") if out is None else out
    bfq.bfq_gemm_block_fp8(d[0], d[1], fmt, d[1].shape[-1], d[2], d[3], out, None)
    return out


def test_gemm_split_k_is_deterministic(cuda_lib, orc):
    """Splits of the K range meet in distributed shared memory and are added in
    a fixed order, so repeated calls agree bit for bit; a workspace is
    accepted and changes nothing.  24 x 512 x 4096 and 200 x 512 x 4096: two
    256-wide output tiles per row tile, K split over a cluster."""
    bfq = cuda_lib
    for M, N, K in ((24, 512, 4096), (200, 512, 4096)):
        assert bfq.bfq_gemm_workspace_bytes(M, N, K) == 0
        aq, sa, wq, sw = _oracle_problem(orc, M, N, K, 0, seed=99 + M)
        d = _to_dev(aq, sa, wq, sw, 0)
        o1 = _no_workspace_gemm(bfq, d, 0)
        o2 = _no_workspace_gemm(bfq, d, 0)
        ws = torch.full((4096,), 0x7F, dtype=torch.uint8, device="cuda")  # accepted, unused
        o3 = bfq.gemm(d[0], d[1], 0, d[2], d[3], workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(o1, o3)
        ref = orc.gemm(aq, sa, 0, wq, sw)
        an, wn = _norms(orc, aq, sa, wq, sw, 0)
        assert_gemm_close(o1.float().cpu().numpy(), ref, an, wn, f"split {M}")


def test_gemm_rejects_format_it_was_not_told(cuda_lib, orc):
    """The scale format travels with the scales: UE8M0 words handed to the GEMM
    as packed give the oracle's result, while the same words handed over as
    fp32 scales give a result far outside the tolerance (the mismatch
    reported in the review of "[Perf] Deepgemm fused layout kernel for
    activations", where packed exponents were read as floats).  The fp32 call
    gets a buffer sized for fp32 scales (the packed words in its first
    columns, zeros after) so that every read stays inside it."""
    bfq = cuda_lib
    M, N, K = 16, 256, 1024
    aq, sa, wq, sw = _oracle_problem(orc, M, N, K, 2, seed=5)
    d = _to_dev(aq, sa, wq, sw, 2)
    good = bfq.gemm(d[0], d[1], 2, d[2], d[3])
    ld = d[1].shape[-1]
    as_f32 = torch.zeros((K // 128, ld), dtype=torch.int32, device="cuda")
    as_f32[:K // 512] = d[1]
    bad = bfq.gemm(d[0], as_f32.view(torch.float32), 0, d[2], d[3])
    torch.cuda.synchronize()
    ref = orc.gemm(aq, sa, 2, wq, sw)
    an, wn = _norms(orc, aq, sa, wq, sw, 2)
    assert_gemm_close(good.float().cpu().numpy(), ref, an, wn, "packed")
    got = bad.float().cpu().numpy()
    with np.errstate(invalid="ignore", over="ignore"):
        err = np.abs(got.astype(np.float64) - ref) / (an[:, None] * wn[None, :])
    assert not (np.isfinite(got).all() and err.max() <= 2e-3), \
        "packed words read as fp32 scales must not pass the tolerance"


SWEEP_NK = [(4096, 7168), (7168, 18432), (18432, 7168), (24576, 1536), (32768, 512),
            (7168, 16384)]
SWEEP_M = [8, 64, 128, 1024, 2048, 4096]


@pytest.mark.slow
@pytest.mark.parametrize("N,K", SWEEP_NK)
def test_gemm_full_size_sweep_sampled(cuda_lib, orc, N, K):
    """The dense shape sweep at full size, in the bench's launch configuration:
    GPU weight quant bit-exact against the oracle, then for every m the GPU
    quant (sampled rows bit-exact) and GEMM (sampled rows within tolerance)."""
    bfq = cuda_lib
    w = synth.weight(N, K, seed=N + K)
    owq, osw = orc.weight_block_quant(bits(w), False)
    wq, sw = bfq.weight_block_quant(w.cuda(), 0)
    torch.cuda.synchronize()
    assert np.array_equal(codes(wq), owq)
    assert np.array_equal(sw.cpu().numpy(), osw)
    wn = np.linalg.norm(orc.dequant_weight(owq, osw), axis=1)
    del w
    for M in SWEEP_M:
        x = synth.activation(M, K, seed=M * 31 + N)
        q, s = bfq.quant(x.cuda(), 0)
        out = bfq.gemm(q, s, 0, wq, sw)
        torch.cuda.synchronize()
        rng = np.random.default_rng(M + N + K)
        rows = np.arange(M) if M <= 8 else np.unique(np.concatenate(
            [[0, M - 1], rng.integers(0, M, 6)]))
        oq, osa = orc.quant(bits(x[torch.from_numpy(rows)]), 0)
        assert np.array_equal(codes(q)[rows], oq)
        assert np.array_equal(scale_np(s, 0)[:, rows], osa[:, :len(rows)])
        ref = orc.gemm(oq, osa, 0, owq, osw)
        an = np.linalg.norm(orc.dequant_rows(oq, osa, 0), axis=1)
        got = out.float().cpu().numpy()[rows]
        assert_gemm_close(got, ref, an, wn, f"sweep m={M} n={N} k={K}")
        assert calc_diff(got, ref) < 1e-4


@pytest.mark.parametrize("fmt", [0, 2])
@pytest.mark.parametrize("M,N,K", [(1152, 4096, 384), (2048, 2560, 512)])
def test_gemm_parity_unsplit_many_tiles(cuda_lib, orc, fmt, M, N, K):
    """Enough tiles that K is not split (one CTA per output tile), with a
    ragged and an odd number of m tiles."""
    bfq = cuda_lib
    assert bfq.bfq_gemm_workspace_bytes(M, N, K) == 0
    aq, sa, wq, sw = _oracle_problem(orc, M, N, K, fmt, seed=M + N + K + fmt)
    d = _to_dev(aq, sa, wq, sw, fmt)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm(d[0], d[1], fmt, d[2], d[3], out=out)
    torch.cuda.synchronize()
    ref = orc.gemm(aq, sa, fmt, wq, sw)
    an, wn = _norms(orc, aq, sa, wq, sw, fmt)
    assert_gemm_close(out.float().cpu().numpy(), ref, an, wn, f"unsplit {M}x{N}x{K}")


@pytest.mark.parametrize("fmt", [0, 2])
@pytest.mark.parametrize("M,N,K", [(40, 13056, 256), (100, 16384, 256)])
def test_gemm_parity_narrow_unsplit_plan(cuda_lib, orc, fmt, M, N, K):
    """One row tile of more than 32 rows whose 256-wide plan would split K
    two ways: the plan takes 128-wide tiles with no split instead."""
    bfq = cuda_lib
    aq, sa, wq, sw = _oracle_problem(orc, M, N, K, fmt, seed=M + N + K + fmt)
    d = _to_dev(aq, sa, wq, sw, fmt)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    _no_workspace_gemm(bfq, d, fmt, out=out)
    torch.cuda.synchronize()
    ref = orc.gemm(aq, sa, fmt, wq, sw)
    an, wn = _norms(orc, aq, sa, wq, sw, fmt)
    assert_gemm_close(out.float().cpu().numpy(), ref, an, wn, f"narrow {M}x{N}x{K}")


@pytest.mark.parametrize("fmt", [0, 2])
@pytest.mark.parametrize("M,N,K", [(1280, 4224, 8192), (1536, 4608, 4096)])
def test_gemm_parity_two_way_split_for_a_partial_second_wave(cuda_lib, orc, fmt, M, N, K):
    """A last wave at most half full.  1280 x 4224 x 8192: 170 tiles of
    128 x 256 (the last column tile half full) with 64 K blocks, so every
    tile's K is split two ways over 2-CTA clusters (340 half-length CTAs)
    instead of a persistent second round.  1536 x 4608 x 4096: 216 tiles
    with 32 K blocks, too short a K for that split, so the persistent kernel
    walks them in two rounds, the second 64 tiles long.  Three sampled rows
    of every row tile, every column."""
    bfq = cuda_lib
    aq, sa, wq, sw = _oracle_problem(orc, M, N, K, fmt, seed=57 + fmt)
    d = _to_dev(aq, sa, wq, sw, fmt)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm(d[0], d[1], fmt, d[2], d[3], out=out)
    out2 = bfq.gemm(d[0], d[1], fmt, d[2], d[3])
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    rng = np.random.default_rng(5 + fmt)
    rows = np.unique(np.concatenate(
        [[t * 128, min(M, t * 128 + 128) - 1, rng.integers(t * 128, min(M, t * 128 + 128))]
         for t in range((M + 127) // 128)]))
    ref = orc.gemm(aq, sa, fmt, wq, sw, rows=rows)
    an, wn = _norms(orc, aq, sa, wq, sw, fmt, rows=rows)
    got = out.float().cpu().numpy()
    assert_gemm_close(got[rows], ref, an, wn, f"two-way split {M}x{N}x{K} fmt{fmt}")
    assert np.isfinite(got).all()


@pytest.mark.parametrize("fmt", [0, 2])
@pytest.mark.parametrize("M,N,K", [(2000, 8192, 256), (2048, 2432, 256), (2048, 2496, 256),
                                   (1100, 5120, 256)])
def test_gemm_parity_persistent_many_tiles(cuda_lib, orc, fmt, M, N, K):
    """More 256-wide tiles than SMs, so the persistent schedule walks several
    tiles per SM.  2000 x 8192: 16 row tiles, the last one ragged, x 32
    column tiles; 2048 x 2432 and 2048 x 2496: the last column tile half and
    three quarters full (two and three of its four staged output boxes
    stored); 1100 x 5120: an odd number of row tiles.  Three sampled rows of
    every row tile against the oracle, every column."""
    bfq = cuda_lib
    assert bfq.bfq_gemm_workspace_bytes(M, N, K) == 0
    aq, sa, wq, sw = _oracle_problem(orc, M, N, K, fmt, seed=31 + fmt + N)
    d = _to_dev(aq, sa, wq, sw, fmt)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm(d[0], d[1], fmt, d[2], d[3], out=out)
    torch.cuda.synchronize()
    rng = np.random.default_rng(fmt)
    rows = np.unique(np.concatenate(
        [[t * 128, min(M, t * 128 + 128) - 1, rng.integers(t * 128, min(M, t * 128 + 128))]
         for t in range((M + 127) // 128)]))
    ref = orc.gemm(aq, sa, fmt, wq, sw, rows=rows)
    an, wn = _norms(orc, aq, sa, wq, sw, fmt, rows=rows)
    got = out.float().cpu().numpy()
    assert_gemm_close(got[rows], ref, an, wn, f"persistent {M}x{N}x{K} fmt{fmt}")
    assert np.isfinite(got).all()


@pytest.mark.parametrize("fmt", [0, 2])
@pytest.mark.parametrize("M,N,K", [(1280, 4096, 512), (2560, 2048, 1024), (2000, 2560, 256)])
def test_gemm_persistent_partial_last_round(cuda_lib, orc, fmt, M, N, K):
    """160 output tiles on a 152-SM part: the persistent schedule's second
    round holds 8 tiles, the last row tiles of the last column tile (the
    2000-row case ends in a ragged row tile).  Every element against the
    oracle."""
    bfq = cuda_lib
    aq, sa, wq, sw = _oracle_problem(orc, M, N, K, fmt, seed=M + N + K + fmt)
    d = _to_dev(aq, sa, wq, sw, fmt)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bfq.gemm(d[0], d[1], fmt, d[2], d[3], out=out)
    torch.cuda.synchronize()
    ref = orc.gemm(aq, sa, fmt, wq, sw)
    an, wn = _norms(orc, aq, sa, wq, sw, fmt)
    assert_gemm_close(out.float().cpu().numpy(), ref, an, wn, f"gemm {M}x{N}x{K} fmt{fmt}")
    assert bfq.bfq_poll_device_status() == 0
