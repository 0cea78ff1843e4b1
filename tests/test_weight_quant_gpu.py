"""128 x 128 block weight quant on the GPU vs the oracle, bit-exact
("vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.1, per_block_cast_to_fp8)."""
import numpy as np
import pytest
import torch

import bfq_synth as synth
from helpers import bits, codes

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("N,K", [(128, 128), (320, 384), (64, 256), (4096, 7168)])
def test_weight_quant_bit_exact(cuda_lib, orc, fmt, N, K):
    bfq = cuda_lib
    w = synth.weight(N, K, seed=N + K)
    wq, sw = bfq.weight_block_quant(w.cuda(), fmt)
    torch.cuda.synchronize()
    owq, osw = orc.weight_block_quant(bits(w), fmt == 1)
    assert np.array_equal(codes(wq), owq)
    assert np.array_equal(sw.cpu().numpy(), osw)


def test_weight_quant_batched_experts(cuda_lib, orc):
    bfq = cuda_lib
    E, N, K = 3, 192, 256  # N % 128 != 0: blocks must not straddle experts
    w = synth.expert_weights(E, N, K, seed=3)
    wq, sw = bfq.weight_block_quant(w.cuda(), 1)
    torch.cuda.synchronize()
    assert sw.shape == (E, 2, 2)
    for e in range(E):
        owq, osw = orc.weight_block_quant(bits(w[e]), True)
        assert np.array_equal(codes(wq[e]), owq)
        assert np.array_equal(sw[e].cpu().numpy(), osw)
