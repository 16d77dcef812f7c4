"""Router, top-6 selection and permutation on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle.reference import margins
from sparse_moe_transformer_03_b300 import flint
from synth import device, gen
from tests.gpu_common import handle_for, layer, to_dev_bf16, x_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    device.build()
    lw = layer(1, 0, True)
    h = handle_for(lw)
    yield lw, h
    flint.flint_moe_destroy(h)


def route(h, T, x=None, logits=None, perm=False):
    idx = torch.empty((T, 6), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 6), dtype=torch.float32, device="cuda")
    off = torch.empty(257, dtype=torch.int32, device="cuda") if perm else None
    gat = torch.empty(T * 6, dtype=torch.int32, device="cuda") if perm else None
    lg = logits if logits is not None else (torch.empty((T, 256), dtype=torch.float32, device="cuda")
                                            if x is not None else None)
    flint.flint_moe_route_only(h, x, lg, T, idx, w, off, gat)
    out = {"idx": idx.cpu().numpy(), "w": w.cpu().numpy()}
    if x is not None:
        out["logits"] = lg.cpu().numpy()
    if perm:
        out["offsets"], out["gather"] = off.cpu().numpy(), gat.cpu().numpy()
    return out


@pytest.mark.parametrize("T", [1, 7, 32, 33, 300, 8192])
def test_selection_from_fed_logits_is_exact(setup, T):
    """Fed the oracle's fp32 logits, the GPU must choose exactly the oracle's
    experts (both rank the same fp32 values) and the permutation must equal
    the oracle's stable counting sort."""
    lw, h = setup
    x = gen.x_gaussian(100 + T, T)
    l64 = oracle.router_logits(x, lw.router_bits(), lw.bias_host())
    l32 = l64.astype(np.float32)
    ref_idx, ref_w = oracle.select(l32.astype(np.float64))
    g = route(h, T, logits=torch.from_numpy(l32).cuda(), perm=True)
    assert np.array_equal(g["idx"], ref_idx)
    assert np.allclose(g["w"], ref_w, rtol=2e-6, atol=1e-7)
    off, gat = oracle.permutation(ref_idx)
    assert np.array_equal(g["offsets"], off)
    assert np.array_equal(g["gather"], gat)


def test_selection_ties_and_extremes(setup):
    _, h = setup
    T = 5
    l = np.zeros((T, 256), np.float32)                 # all equal: experts 0..5
    l[1, [250, 3, 77, 200, 9, 100, 101]] = 3.0         # seven equal maxima
    l[2] = -np.arange(256, dtype=np.float32)           # strictly decreasing
    l[3] = np.float32(60.0) - np.arange(256, dtype=np.float32) * 1e-3  # sigmoid saturates at 1
    l[4] = np.random.default_rng(4).normal(0, 1, 256).astype(np.float32)
    ref_idx, ref_w = oracle.select(l.astype(np.float64))
    g = route(h, T, logits=torch.from_numpy(l).cuda(), perm=True)
    assert np.array_equal(g["idx"], ref_idx)
    assert g["idx"][0].tolist() == [0, 1, 2, 3, 4, 5]
    assert g["idx"][1].tolist() == [3, 9, 77, 100, 101, 200]
    assert g["idx"][3].tolist() == [0, 1, 2, 3, 4, 5]
    assert np.allclose(g["w"], ref_w, rtol=2e-6, atol=1e-7)
    assert np.allclose(g["w"].sum(1), 1.0, atol=1e-6)


@pytest.mark.parametrize("T,kind", [(1, "gauss"), (4, "gauss"), (32, "clustered"), (100, "gauss")])
def test_router_logits_and_selection_from_x(setup, T, kind):
    lw, h = setup
    xb = x_for(kind, 200 + T, T)
    l64 = oracle.router_logits(xb, lw.router_bits(), lw.bias_host())
    ref_idx, _ = oracle.select(l64)
    g = route(h, T, x=to_dev_bf16(xb), perm=True)
    # fp32 accumulation of 2048 bf16 products: |error| well below 1e-4
    assert np.abs(g["logits"] - l64).max() < 1e-4
    near = margins(l64) < 1e-5
    for t in range(T):
        if near[t]:
            assert set(g["idx"][t][:5]) == set(ref_idx[t][:5])
        else:
            assert g["idx"][t].tolist() == ref_idx[t].tolist()
    # the permutation of the GPU's own choice is a valid stable counting sort
    off = g["offsets"]
    assert off[0] == 0 and off[-1] == 6 * T and np.all(np.diff(off) >= 0)
    flat = g["idx"].ravel()
    assert np.array_equal(g["gather"], np.argsort(flat, kind="stable"))
