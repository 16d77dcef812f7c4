"""Prefill path (T > 32, tcgen05 grouped GEMMs) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from oracle.reference import LayerOracle, compare
from sparse_moe_transformer_03_b300 import flint
from synth import device, gen
from tests.gpu_common import handle_for, layer, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    device.build()
    lw = layer(1, 0, True)          # layer 0 of the decode stack: skewed router bias
    h = handle_for(lw)
    yield lw, h, LayerOracle.from_bf16_layer(lw)
    flint.flint_moe_destroy(h)


def run(h, xb):
    x = to_dev_bf16(xb)
    y = torch.full_like(x, float("nan"))
    flint.flint_moe_forward(h, x, xb.shape[0], y)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("T", [33, 57, 200])
def test_prefill_small_full_compare(setup, T):
    lw, h, orc = setup
    xb = gen.x_gaussian(400 + T, T)
    y = run(h, xb).float().cpu().numpy()
    assert np.isfinite(y).all()
    ref, alt = orc.forward_with_alternatives(xb)
    res = compare(y, ref, alt)
    assert res["ok"], res


def full_compare(orc, xb, y):
    """Every row of the device output against the oracle, element by element."""
    ref, alt = orc.forward_with_alternatives(xb)
    res = compare(y.float().cpu().numpy(), ref, alt)
    assert res["ok"], res
    return res


def test_prefill_1000_tokens(setup):
    lw, h, orc = setup
    xb = gen.x_gaussian(14, 1000)
    y = run(h, xb)
    assert torch.isfinite(y.float()).all()
    full_compare(orc, xb, y)


def test_prefill_8192_tokens_full_config(setup):
    """The prefill workload: 8192 tokens, x ~ N(0,1) RMS-normalised (seed 14),
    skewed router bias.  All 8192 rows are compared with the oracle (so every
    expert's every 256-token pass and its ragged last pass is covered), and
    a second forward is bit-identical (every sum runs in a fixed order)."""
    lw, h, orc = setup
    xb = gen.x_gaussian(14, 8192)
    y = run(h, xb)
    assert torch.isfinite(y.float()).all()
    full_compare(orc, xb, y)
    y2 = run(h, xb)
    assert torch.equal(y2, y)


def test_prefill_chunked_beyond_8192(setup):
    """8269 tokens: one full 8192-token chunk and a ragged 77-token chunk,
    every row compared."""
    lw, h, orc = setup
    T = 8192 + 77
    xb = gen.x_gaussian(15, T)
    y = run(h, xb)
    assert torch.isfinite(y.float()).all()
    full_compare(orc, xb, y)
