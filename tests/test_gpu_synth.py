"""The CUDA input generator draws the same numbers as the numpy one."""
import numpy as np
import pytest
import torch

from synth import device, gen

pytestmark = pytest.mark.gpu


def test_device_generator_matches_host():
    device.build()
    n = 1 << 20
    t = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    device.fill_normal_bf16(t, 3, 5, gen.gate_up_tensor(9), 0.02)
    host = gen.normal_bf16(3, 5, gen.gate_up_tensor(9), (n,), 0.02)
    dev = t.view(torch.int16).cpu().numpy().view(np.uint16)
    diff = dev != host
    # double-precision log/cos/sin may differ in the last ulp between libm and
    # CUDA; after rounding to bf16 that almost never shows
    assert diff.sum() <= 2, diff.sum()
    # an offset window
    t2 = torch.empty(1001, dtype=torch.bfloat16, device="cuda")
    device.fill_normal_bf16(t2, 3, 5, gen.gate_up_tensor(9), 0.02, start=12345)
    assert (t2.view(torch.int16).cpu().numpy().view(np.uint16) != host[12345:13346]).sum() <= 1
    b = torch.empty(256, dtype=torch.float32, device="cuda")
    device.fill_normal_f32(b, 1, 0, gen.T_ROUTER_B, gen.BIAS_STD)
    assert np.allclose(b.cpu().numpy(), gen.router_bias(1, 0), rtol=1e-6, atol=0)


def test_batched_generator_matches_per_tensor():
    device.build()
    t = torch.empty((3, 64, 32), dtype=torch.bfloat16, device="cuda")
    device.fill_normal_bf16_batched(t, 2, 4, gen.gate_up_tensor(5), 2, 0.02)
    for i in range(3):
        host = gen.normal_bf16(2, 4, gen.gate_up_tensor(5 + i), (64 * 32,), 0.02)
        got = t[i].reshape(-1).view(torch.int16).cpu().numpy().view(np.uint16)
        assert (got != host).sum() <= 1
