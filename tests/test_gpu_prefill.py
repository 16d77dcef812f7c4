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


def sample_compare(orc, xb, y, rows):
    sub = xb[rows]
    ref, alt = orc.forward_with_alternatives(sub)
    res = compare(y[rows].float().cpu().numpy(), ref, alt)
    assert res["ok"], res
    return res


def test_prefill_1000_tokens(setup):
    lw, h, orc = setup
    xb = gen.x_gaussian(14, 1000)
    y = run(h, xb)
    assert torch.isfinite(y.float()).all()
    rows = np.concatenate([np.arange(0, 1000, 37), [999]])
    sample_compare(orc, xb, y, rows)


def test_prefill_8192_tokens_full_config(setup):
    """The prefill workload: 8192 tokens, x ~ N(0,1) RMS-normalised (seed 14),
    skewed router bias; sampled rows across every 128-token block and the
    last one, compared with the oracle token by token."""
    lw, h, orc = setup
    xb = gen.x_gaussian(14, 8192)
    y = run(h, xb)
    assert torch.isfinite(y.float()).all()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, 8192, 128) + rng.integers(0, 128, 64), [0, 8191]]))
    sample_compare(orc, xb, y, rows)
    # deterministic: every sum runs in a fixed order
    y2 = run(h, xb)
    assert torch.equal(y2, y)


def test_prefill_chunked_beyond_8192(setup):
    lw, h, orc = setup
    T = 8192 + 77
    xb = gen.x_gaussian(15, T)
    y = run(h, xb)
    assert torch.isfinite(y.float()).all()
    rows = np.array([0, 5000, 8191, 8192, 8200, T - 1])
    sample_compare(orc, xb, y, rows)
