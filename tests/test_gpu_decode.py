"""Decode path (T <= 32) of flint_moe_forward against the fp64 oracle."""
import numpy as np
import pytest
import torch

from oracle.reference import LayerOracle, compare
from sparse_moe_transformer_03_b300 import flint
from synth import device
from tests.gpu_common import handle_for, layer, to_dev_bf16, x_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=[(0, 0, False), (1, 0, True)], ids=["seed0", "seed1-bias"])
def setup(request):
    device.build()
    lw = layer(*request.param)
    h = handle_for(lw)
    yield lw, h, LayerOracle.from_bf16_layer(lw)
    flint.flint_moe_destroy(h)


def forward(h, xb):
    T = xb.shape[0]
    x = to_dev_bf16(xb)
    y = torch.full_like(x, float("nan"))
    flint.flint_moe_forward(h, x, T, y)
    torch.cuda.synchronize()
    return y.float().cpu().numpy()


@pytest.mark.parametrize("T,kind", [(1, "gauss"), (2, "gauss"), (4, "gauss"), (8, "clustered"),
                                    (17, "clustered"), (32, "clustered"), (32, "gauss")])
def test_decode_matches_oracle(setup, T, kind):
    lw, h, orc = setup
    xb = x_for(kind, 300 + T, T)
    y = forward(h, xb)
    assert np.isfinite(y).all()
    ref, alt = orc.forward_with_alternatives(xb)
    res = compare(y, ref, alt)
    assert res["ok"], res


def test_decode_is_deterministic_and_repeatable(setup):
    lw, h, _ = setup
    xb = x_for("clustered", 77, 32)
    y1 = forward(h, xb)
    y2 = forward(h, xb)
    assert np.array_equal(y1, y2)


def test_forward_argument_checks(setup):
    _, h, _ = setup
    x = torch.zeros((4, 2048), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros_like(x)
    lib = flint.load_library()
    import ctypes
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    hh = ctypes.c_void_p(h)
    assert lib.flint_moe_forward(hh, ctypes.c_void_p(x.data_ptr() + 2), 4, ctypes.c_void_p(y.data_ptr()), s) == 1
    assert lib.flint_moe_forward(hh, ctypes.c_void_p(x.data_ptr()), 0, ctypes.c_void_p(y.data_ptr()), s) == 1
    assert lib.flint_moe_forward(hh, ctypes.c_void_p(x.data_ptr()), 4, ctypes.c_void_p(x.data_ptr() + 4096), s) == 1


def test_bounded_wait_gives_up_with_status():
    # a wait on a barrier nothing arrives on returns FLINT_ERR_DEVICE_TIMEOUT
    assert flint.flint_debug_bounded_wait(2_000_000) == 4
    torch.cuda.synchronize()


def test_bf16_expert_buffers_are_not_read_after_create():
    """The handle's tiled copy is the only expert storage both paths read: the
    caller's bf16 expert buffers, overwritten with NaN right after create,
    change nothing (decode sizes and the many-token path)."""
    device.build()
    own = device.LayerWeights(0, 0, False)
    h = handle_for(own)
    try:
        own.gate_up.fill_(float("nan"))
        own.down.fill_(float("nan"))
        torch.cuda.synchronize()
        orc = LayerOracle.from_bf16_layer(layer(0, 0, False))
        for T in (1, 8, 32, 40):
            xb = x_for("clustered", 500 + T, T)
            y = forward(h, xb)
            assert np.isfinite(y).all(), T
            ref, alt = orc.forward_with_alternatives(xb)
            res = compare(y, ref, alt)
            assert res["ok"], (T, res)
    finally:
        flint.flint_moe_destroy(h)
        del own
        torch.cuda.empty_cache()
