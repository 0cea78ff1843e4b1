"""The debug build (libbfq_debug.so, compiled with BFQ_DEVICE_CHECKS): every
kernel checks each global offset it computes against the extent of its
array, as the host derived it from the call's arguments, and latches
BFQ_ERR_DEVICE_BOUNDS instead of making the access.  compute-sanitizer is
not available, so this is the library's own out-of-bounds detector.

A subprocess loads the debug build and runs one case of every kernel and
launch plan (quant in three formats, weight quant, silu-mul-quant, dense
GEMM split over a cluster / unsplit / persistent / with fused output quant,
masked GEMM per-tile and persistent, both fused silu up projections, the
block-scaled dense and masked GEMMs).  No check may fire, and every output
must equal the release build's bit for bit (the checks change no
arithmetic)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_cases(bfq):
    """Outputs (as numpy bytes) of one case per kernel and plan; inputs seeded."""
    import bfq_synth as synth

    dev = torch.device("cuda", 0)
    outs = {}

    def keep(name, t):
        outs[name] = t.detach().contiguous().view(torch.uint8).cpu().numpy().copy()

    x = synth.activation(200, 1152, seed=1, device=dev)
    for fmt in (0, 1, 2):
        q, s = bfq.quant(x, fmt)
        keep(f"quant{fmt}_q", q)
        keep(f"quant{fmt}_s", s[:, :200])
    w = synth.expert_weights(2, 320, 384, seed=2, device=dev)
    for fmt in (0, 1):
        wq, sw = bfq.weight_block_quant(w, fmt)
        keep(f"wquant{fmt}_q", wq)
        keep(f"wquant{fmt}_s", sw)
    counts = torch.tensor([70, 0, 136], dtype=torch.int32, device=dev)
    xs = synth.masked_activation(3, 136, 768, counts.cpu(), seed=3, device=dev, poison=False)
    for fmt in (0, 2):
        q, s = bfq.silu_mul_quant(xs, counts, fmt)
        for e, c in enumerate((70, 0, 136)):
            keep(f"silu{fmt}_q{e}", q[e, :c])
            keep(f"silu{fmt}_s{e}", s[e, :, :c])
    # dense GEMM plans: K split over a cluster, unsplit tiles, persistent
    for (m, n, k) in ((40, 1024, 2048), (1024, 8192, 256), (2048, 2560, 256)):
        a, sa = bfq.quant(synth.activation(m, k, seed=m + n, device=dev), 0)
        wq, sw = bfq.weight_block_quant(synth.weight(n, k, seed=m + n + 1, device=dev), 0)
        keep(f"gemm{m}x{n}x{k}", bfq.gemm(a, sa, 0, wq, sw))
        if n % 128 == 0:
            q2, s2 = bfq.gemm_quant(a, sa, 0, wq, sw, 2)
            keep(f"gemmq{m}x{n}x{k}_q", q2)
            keep(f"gemmq{m}x{n}x{k}_s", s2[:, :m])
    # masked GEMM: 128-wide per-tile plan and the persistent plan
    E, T, K = 3, 136, 384
    am = torch.zeros((E, T, K), dtype=torch.float8_e4m3fn, device=dev)
    sam = torch.zeros((E, bfq.scale_cols(K, 2), T), dtype=torch.int32, device=dev)
    xm = synth.masked_activation(E, T, K, counts.cpu(), seed=4, device=dev, poison=False)
    for e, c in enumerate((70, 0, 136)):
        if c:
            bfq.bfq_quant(xm[e, :c], am[e, :c], sam[e], 2, T)
    for n in (128, 320):
        wm, swm = bfq.weight_block_quant(synth.expert_weights(E, n, K, seed=5 + n, device=dev), 1)
        out = torch.zeros((E, T, n), dtype=torch.bfloat16, device=dev)
        bfq.gemm_masked(am, sam, 2, wm, swm, counts, out=out)
        keep(f"masked{n}", out)
        if n == 320:
            outb = torch.zeros((E, T, n), dtype=torch.bfloat16, device=dev)
            bfq.gemm_masked_ue8m0(am, sam, 2, wm, swm, counts, out=outb)
            keep("masked_bs", outb)
    # fused silu up projections (promotion and block-scaled)
    wu, swu = bfq.weight_block_quant(synth.expert_weights(E, 512, K, seed=6, device=dev), 1)
    wi, si = bfq.interleave_gate_up(wu, swu)
    fq, fs = bfq.gemm_masked_silu_quant(am, sam, 2, wi, si, counts, 2)
    q_b = torch.zeros((E, T, 256), dtype=torch.float8_e4m3fn, device=dev)
    s_b = torch.zeros((E, bfq.scale_cols(256, 2), T), dtype=torch.int32, device=dev)
    bfq.bfq_gemm_block_fp8_masked_silu_quant_ue8m0(am, sam, 2, T, wi, si, counts, 2, q_b, s_b, T)
    for e, c in enumerate((70, 0, 136)):
        keep(f"fused_q{e}", fq[e, :c])
        keep(f"fused_s{e}", fs[e, :, :c])
        keep(f"fused_bs_q{e}", q_b[e, :c])
        keep(f"fused_bs_s{e}", s_b[e, :, :c])
    # block-scaled dense GEMM on its own plan
    a, sa = bfq.quant(synth.activation(1024, 1024, seed=7, device=dev), 2)
    wq, sw = bfq.weight_block_quant(synth.weight(8192, 1024, seed=8, device=dev), 1)
    keep("gemm_bs", bfq.gemm_ue8m0(a, sa, 2, wq, sw))
    torch.cuda.synchronize()
    outs["status"] = np.array([bfq.bfq_poll_device_status()], np.int32)
    return outs


_SCRIPT = r"""
import sys
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np
import block_scaled_fp8_quant_gb300 as bfq
bfq.load_library(debug=True)
from test_debug_build_gpu import run_cases
np.savez(sys.argv[2], **run_cases(bfq))
"""


def test_debug_build_fires_no_check_and_matches_release(cuda_lib, tmp_path):
    path = str(tmp_path / "debug_outs.npz")
    r = subprocess.run([sys.executable, "-c", _SCRIPT, ROOT, path], capture_output=True,
                       text=True, timeout=1500, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    dbg = np.load(path)
    assert int(dbg["status"][0]) == 0, f"debug build latched status {int(dbg['status'][0])}"
    rel = run_cases(cuda_lib)
    assert int(rel["status"][0]) == 0
    assert set(dbg.files) == set(rel)
    for name in rel:
        assert np.array_equal(dbg[name], rel[name]), f"{name}: debug and release builds differ"
