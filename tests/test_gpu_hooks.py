"""The per-kernel event hook: events bracket exactly the named kernel."""
import pytest
import torch

from sparse_moe_transformer_03_b300 import flint
from synth import device, gen
from tests.gpu_common import handle_for, layer, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,kernels", [(4, (0, 1, 2)), (300, (0, 1, 2, 3))])
def test_kernel_events_time_each_kernel(T, kernels):
    device.build()
    lw = layer(1, 0, True)
    h = handle_for(lw)
    try:
        x = to_dev_bf16(gen.x_gaussian(7, T))
        y = torch.empty_like(x)
        y_ref = torch.empty_like(x)
        flint.flint_moe_forward(h, x, T, y_ref)
        s = torch.cuda.current_stream()
        for k in kernels:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flint.flint_moe_set_kernel_events(h, k, e0, e1)
            flint.flint_moe_forward(h, x, T, y)
            e1.synchronize()
            ms = e0.elapsed_time(e1)
            assert 0.0 < ms < 100.0
            assert torch.equal(y, y_ref)          # the hook changes no result
        flint.flint_moe_set_kernel_events(h, -1)
        with pytest.raises(flint.FlintError):
            flint.flint_moe_set_kernel_events(h, 7, e0, e1)
    finally:
        flint.flint_moe_destroy(h)
