"""flint_permute_static (the permutation with a fixed device scratch array)
against the oracle's stable counting sort and against flint_moe_route_only's
permutation, through the C ABI.  Kept in a file collected last so that it
also runs after every other GPU test."""
import numpy as np
import pytest
import torch

import oracle

from sparse_moe_transformer_03_b300 import flint
from synth import device, gen
from tests.gpu_common import handle_for, layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    device.build()
    hd = handle_for(layer(1, 0, True))
    yield hd
    flint.flint_moe_destroy(hd)


def _route(h, T, seed):
    """idx, offsets, gather of route_only on fed logits (its existing path)."""
    rng = np.random.default_rng(seed)
    logits = torch.from_numpy(rng.normal(0, 1, (T, 256)).astype(np.float32)).cuda()
    idx = torch.empty((T, 6), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 6), dtype=torch.float32, device="cuda")
    off = torch.empty(257, dtype=torch.int32, device="cuda")
    gat = torch.empty(T * 6, dtype=torch.int32, device="cuda")
    flint.flint_moe_route_only(h, None, logits, T, idx, w, off, gat)
    return idx, off.cpu(), gat.cpu()


def _static(idx, T):
    off = torch.full((257,), -7, dtype=torch.int32, device="cuda")
    gat = torch.full((T * 6,), -7, dtype=torch.int32, device="cuda")
    flint.flint_permute_static(idx, T, off, gat)
    return off.cpu(), gat.cpu()


@pytest.mark.parametrize("Ts", [(8192, 8192), (8192, 37), (1, 300)])
def test_static_scratch_matches_route_only_two_calls(h, Ts):
    """Two calls in a row (the second reuses the scratch the first left behind)."""
    for n, T in enumerate(Ts):
        idx, off_ref, gat_ref = _route(h, T, seed=1000 * n + T)
        off, gat = _static(idx, T)
        assert torch.equal(off, off_ref)
        assert torch.equal(gat, gat_ref)
        off_o, gat_o = oracle.permutation(idx.cpu().numpy())
        assert np.array_equal(off.numpy(), off_o)
        assert np.array_equal(gat.numpy(), gat_o)


def test_static_scratch_rejects_beyond_maximum():
    idx = torch.zeros((8193, 6), dtype=torch.int32, device="cuda")
    off = torch.empty(257, dtype=torch.int32, device="cuda")
    gat = torch.empty(8193 * 6, dtype=torch.int32, device="cuda")
    with pytest.raises(flint.FlintError) as ei:
        flint.flint_permute_static(idx, 8193, off, gat)
    assert ei.value.code == 1   # FLINT_ERR_INVALID_ARG


def test_static_scratch_bad_index_then_recovers(h):
    """An id outside 0..255 is reported, and the next call succeeds."""
    T = 64
    idx = torch.zeros((T, 6), dtype=torch.int32, device="cuda")
    idx[:, :] = torch.arange(6, dtype=torch.int32, device="cuda")
    idx[5, 2] = 300
    off = torch.empty(257, dtype=torch.int32, device="cuda")
    gat = torch.empty(T * 6, dtype=torch.int32, device="cuda")
    with pytest.raises(flint.FlintError) as ei:
        flint.flint_permute_static(idx, T, off, gat)
    assert ei.value.code == 5   # FLINT_ERR_DEVICE_BADINDEX
    idx2, off_ref, gat_ref = _route(h, T, seed=5)
    off2, gat2 = _static(idx2, T)
    assert torch.equal(off2, off_ref) and torch.equal(gat2, gat_ref)
