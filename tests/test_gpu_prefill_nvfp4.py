"""NVFP4 (W4A16) many-token path of flint_moe_forward (T > 32: the grouped
tcgen05 GEMMs whose weight tiles are dequantised from the owned NVFP4 layout
in shared memory) against the fp64 oracle run on the same NVFP4 codes,
every output row compared."""
import numpy as np
import pytest
import torch

from oracle.reference import compare
from sparse_moe_transformer_03_b300 import flint
from synth import device, gen
from tests.gpu_common import layer, nvfp4_oracle, to_dev_bf16, x_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    device.build()
    lw = layer(1, 0, True)          # layer 0 of the decode stack: skewed router bias
    q = device.LayerNVFP4(lw)
    gu, dn, sh = q.create_args()
    h = flint.flint_moe_create(lw.router_W, lw.router_b, gu, dn, sh, dtype=flint.FLINT_NVFP4)
    yield lw, q, h, nvfp4_oracle(lw, q)
    flint.flint_moe_destroy(h)


def run(h, xb):
    x = to_dev_bf16(xb)
    y = torch.full_like(x, float("nan"))
    flint.flint_moe_forward(h, x, xb.shape[0], y)
    torch.cuda.synchronize()
    return y


def full_compare(orc, xb, y):
    yf = y.float().cpu().numpy()
    assert np.isfinite(yf).all()
    ref, alt = orc.forward_with_alternatives(xb)
    res = compare(yf, ref, alt)
    assert res["ok"], res
    return res


@pytest.mark.parametrize("T,kind", [(33, "gauss"), (57, "clustered"), (200, "gauss"), (1000, "clustered")])
def test_nvfp4_prefill_matches_oracle(setup, T, kind):
    """Above the decode limit: one token pass per expert (T = 33) up to
    experts with several 256-token passes (clustered tokens at T = 1000)."""
    lw, q, h, orc = setup
    xb = x_for(kind, 700 + T, T)
    full_compare(orc, xb, run(h, xb))


def test_nvfp4_prefill_8192_tokens_full_config(setup):
    """The 8192-token prefill of the NVFP4 layer (x ~ N(0,1) RMS-normalised,
    seed 14, skewed router bias): all rows against the oracle, and a second
    forward bit-identical."""
    lw, q, h, orc = setup
    xb = gen.x_gaussian(14, 8192)
    y = run(h, xb)
    full_compare(orc, xb, y)
    assert torch.equal(run(h, xb), y)


def test_nvfp4_prefill_chunked_beyond_8192(setup):
    """8269 tokens: a full 8192-token chunk, then a ragged 77-token one."""
    lw, q, h, orc = setup
    xb = gen.x_gaussian(15, 8192 + 77)
    full_compare(orc, xb, run(h, xb))


def test_nvfp4_prefill_then_decode_on_one_handle(setup):
    """The two NVFP4 paths share the handle's workspace: a prefill, a decode
    and the prefill again give the oracle's answer and identical repeats."""
    lw, q, h, orc = setup
    xa = gen.x_gaussian(16, 300)
    xb = x_for("clustered", 17, 8)
    ya = run(h, xa)
    yb = run(h, xb)
    assert torch.equal(run(h, xa), ya)
    full_compare(orc, xb, yb)
