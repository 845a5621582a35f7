"""The device-side timeout path, exercised without a fault: moe_watchdog_selftest waits on
an mbarrier that nothing completes through the GEMM kernels' bounded wait; the status word
must then read MOE_ERR_TIMEOUT, the read must clear it, and the context must stay usable."""
import time

import numpy as np
import pytest
import torch

import oracle
from deepseek_moe_layer_gb300 import binding

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_watchdog_timeout_is_reported_and_cleared():
    binding.device_status()  # start clean
    t0 = time.perf_counter()
    binding.watchdog_selftest(20_000_000)  # 20 ms
    with pytest.raises(binding.MoeError) as e:
        binding.device_status()
    assert e.value.code == binding.MOE_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.02  # the wait ran its limit before giving up
    binding.device_status()  # the read above cleared the word


def test_context_usable_after_timeout():
    binding.watchdog_selftest(1_000_000)
    with pytest.raises(binding.MoeError):
        binding.device_status()
    g = torch.Generator(device=DEV).manual_seed(1)
    logits = torch.randn(64, 32, generator=g, device=DEV)
    gi, gs = binding.route_softmax(logits, 4)
    torch.cuda.synchronize()
    binding.device_status()
    ri, rs = oracle.route_softmax(logits.cpu().numpy(), 4)
    assert np.array_equal(gi.cpu().numpy(), ri)
