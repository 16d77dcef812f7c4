"""NVFP4 (W4A16) decode path of flint_moe_forward against the fp64 oracle run
on the same NVFP4 weights (decoded exactly), and the device NVFP4 encoder of
the input generator against the host one."""
import numpy as np
import pytest
import torch

import oracle
from oracle.reference import compare
from sparse_moe_transformer_03_b300 import flint
from synth import device, gen
from tests.gpu_common import nvfp4_oracle, layer, to_dev_bf16, x_for

pytestmark = pytest.mark.gpu



@pytest.fixture(scope="module", params=[(0, 0, False), (1, 0, True)], ids=["seed0", "seed1-bias"])
def setup(request):
    device.build()
    lw = layer(*request.param)
    q = device.LayerNVFP4(lw)
    gu, dn, sh = q.create_args()
    h = flint.flint_moe_create(lw.router_W, lw.router_b, gu, dn, sh, dtype=flint.FLINT_NVFP4)
    yield lw, q, h, nvfp4_oracle(lw, q)
    flint.flint_moe_destroy(h)


def forward(h, xb):
    T = xb.shape[0]
    x = to_dev_bf16(xb)
    y = torch.full_like(x, float("nan"))
    flint.flint_moe_forward(h, x, T, y)
    torch.cuda.synchronize()
    return y.float().cpu().numpy()


def test_device_encoder_matches_host_encoder():
    device.build()
    lw = layer(0, 0, False)
    for e in (3, 256):
        gu, dn = lw.expert_bits(e)
        for bits, dev in ((gu, lw.gate_up[e:e + 1]), (dn, lw.down[e:e + 1])):
            pk_h, sc_h, ts_h = gen.nvfp4_quantize(bits)
            pk_d, sc_d, ts_d = device.nvfp4_quantize(dev.contiguous())
            assert np.array_equal(pk_d[0].cpu().numpy(), pk_h)
            assert np.array_equal(sc_d[0].cpu().numpy(), sc_h)
            assert ts_d[0].item() == float(ts_h)


@pytest.mark.parametrize("T,kind", [(1, "gauss"), (4, "gauss"), (8, "clustered"), (17, "clustered"),
                                    (32, "clustered"), (32, "gauss"), (45, "gauss")])
def test_nvfp4_decode_matches_oracle(setup, T, kind):
    lw, q, h, orc = setup
    xb = x_for(kind, 500 + T, T)
    y = forward(h, xb)
    assert np.isfinite(y).all()
    ref, alt = orc.forward_with_alternatives(xb)
    res = compare(y, ref, alt)
    assert res["ok"], res


def test_nvfp4_two_calls_in_a_row_and_determinism(setup):
    lw, q, h, orc = setup
    xa = x_for("clustered", 91, 32)
    xb = x_for("gauss", 92, 3)
    ya1 = forward(h, xa)
    yb = forward(h, xb)
    ya2 = forward(h, xa)
    assert np.array_equal(ya1, ya2)
    ref, alt = orc.forward_with_alternatives(xb)
    assert compare(yb, ref, alt)["ok"]


def test_nvfp4_routing_is_the_bf16_routing(setup):
    """The router stays bf16: route-only on an NVFP4 handle equals the oracle's selection."""
    lw, q, h, orc = setup
    T = 16
    xb = gen.x_gaussian(93, T)
    l64 = oracle.router_logits(xb, lw.router_bits(), lw.bias_host())
    ref_idx, _ = oracle.select(l64.astype(np.float32).astype(np.float64))
    idx = torch.empty((T, 6), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 6), dtype=torch.float32, device="cuda")
    flint.flint_moe_route_only(h, None, torch.from_numpy(l64.astype(np.float32)).cuda(), T, idx, w)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
