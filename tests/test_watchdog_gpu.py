"""The kernel watchdog: a bounded wait that runs out records BFQ_ERR_TIMEOUT
in the device latch, the kernel returns, and the context stays usable."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_watchdog_times_out_and_context_survives(cuda_lib):
    bfq = cuda_lib
    assert bfq.bfq_poll_device_status() == 0
    bfq.bfq_watchdog_selftest(2000)  # 2 ms on a barrier nothing completes
    assert bfq.bfq_poll_device_status() == 6  # BFQ_ERR_TIMEOUT
    assert bfq.bfq_poll_device_status() == 0  # the latch was cleared
    x = torch.ones((4, 128), dtype=torch.bfloat16, device="cuda")
    q, s = bfq.quant(x, 0)
    torch.cuda.synchronize()
    assert q.view(torch.uint8).eq(0x7E).all().item()  # 1.0 / (1/448) -> 448
