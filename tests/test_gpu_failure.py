"""Failure detection on the GPU without faulting it: a bounded wait on a
barrier that nothing completes must give up and report MOE_ERR_TIMEOUT, and
the context must stay usable afterwards."""
import torch

from gpu_helpers import gpu, require_gpu


@gpu
def test_bounded_wait_reports_timeout_and_context_survives():
    require_gpu()
    from sparse_moe_layer_13_b300 import binding
    assert binding.selftest_wait_timeout(2000) == 5          # MOE_ERR_TIMEOUT after ~2 ms
    binding.check_device_status()                            # cleared
    x = torch.randn(64, 256, device="cuda").to(torch.bfloat16)
    q, s = binding.quant_1x128(x)                            # the context still runs kernels
    binding.check_device_status()
    assert torch.all(s > 0)
