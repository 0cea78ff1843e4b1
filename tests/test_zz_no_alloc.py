"""bfq_gemm_block_fp8_noalloc: the GEMM for callers that cannot allocate device
memory (plugins in frameworks that own all device memory, serving loops that
forbid allocation after start-up).  No launch plan needs
scratch (K splits reduce through distributed shared memory).

The test calls it through the C ABI twice in a row, on shapes whose launch
plan splits K and on one that does not, and compares each result with the
regular entry point's output on the same inputs, within the GEMM tolerance
of the other tests.  This file is collected last so a failure here cannot hide others."""
import ctypes

import numpy as np
import pytest
import torch

import bfq_synth as synth
from helpers import assert_gemm_close, bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,fmt", [(24, 512, 4096, 0), (8, 4096, 7168, 0),
                                       (100, 1024, 2048, 2), (1024, 4096, 1024, 0)])
def test_noalloc_matches_workspace_entry_point(cuda_lib, orc, M, N, K, fmt):
    bfq = cuda_lib
    lib = bfq.load_library()
    assert lib.bfq_gemm_noalloc_scratch_bytes() == 0 == bfq.bfq_gemm_workspace_bytes(M, N, K)
    x = synth.activation(M, K, seed=M + N + K)
    w = synth.weight(N, K, seed=M + N + K + 1)
    aq, sa = orc.quant(bits(x), fmt)
    wq, sw = orc.weight_block_quant(bits(w), fmt != 0)
    d_aq = torch.from_numpy(aq).cuda().view(torch.float8_e4m3fn)
    d_sa = torch.from_numpy(sa.view(np.int32) if fmt == 2 else sa).cuda()
    d_wq = torch.from_numpy(wq).cuda().view(torch.float8_e4m3fn)
    d_sw = torch.from_numpy(sw).cuda()

    ref = bfq.gemm(d_aq, d_sa, fmt, d_wq, d_sw)  # regular entry point
    torch.cuda.synchronize()
    ref_h = ref.float().cpu().numpy().astype(np.float64)
    an = np.linalg.norm(orc.dequant_rows(aq, sa, fmt), axis=1)
    wn = np.linalg.norm(orc.dequant_weight(wq, sw), axis=1)

    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = lib.bfq_gemm_block_fp8_noalloc(
            ctypes.c_void_p(d_aq.data_ptr()), ctypes.c_void_p(d_sa.data_ptr()), fmt,
            d_sa.shape[-1], ctypes.c_void_p(d_wq.data_ptr()), ctypes.c_void_p(d_sw.data_ptr()),
            M, N, K, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(stream))
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert_gemm_close(out.float().cpu().numpy(), ref_h, an, wn, f"noalloc call {call}")
    assert bfq.bfq_poll_device_status() == 0
