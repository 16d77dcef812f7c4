"""The 47-layer NVFP4 (W4A16) decode stack at full size in the benchmark's
launch configuration (the 47 forwards captured into one CUDA graph and
replayed), every layer checked against the fp64 oracle run on the same NVFP4
codes, at T = 1 and 32."""
import numpy as np
import pytest
import torch

from oracle.reference import compare
from sparse_moe_transformer_03_b300 import flint
from synth import device, gen
from tests.gpu_common import nvfp4_oracle
from tests.test_gpu_stack import replay_stack

pytestmark = pytest.mark.gpu

N_LAYERS = 47


@pytest.fixture(scope="module")
def stack():
    device.build()
    layers, handles = [], []
    for l in range(N_LAYERS):
        lw = device.LayerWeights(1, l, True)
        q = device.LayerNVFP4(lw)
        gu, dn, sh = q.create_args()
        handles.append(flint.flint_moe_create(lw.router_W, lw.router_b, gu, dn, sh, dtype=flint.FLINT_NVFP4))
        lw.gate_up = lw.down = None          # the handle owns its repacked copy; the router stays borrowed
        layers.append((lw, q))
    torch.cuda.empty_cache()
    yield layers, handles
    for h in handles:
        flint.flint_moe_destroy(h)
    del layers
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T,kind,seed", [(1, "gauss", 11), (32, "clustered", 13)])
def test_nvfp4_stack_graph_replay_matches_oracle(stack, T, kind, seed):
    layers, handles = stack
    xb = gen.x_gaussian(seed, T) if kind == "gauss" else gen.x_clustered(seed, T)[0]
    ys = replay_stack(handles, xb, T)
    for l in range(N_LAYERS):
        assert np.isfinite(ys[l]).all(), l
        ref, alt = nvfp4_oracle(*layers[l]).forward_with_alternatives(xb)
        res = compare(ys[l], ref, alt)
        assert res["ok"], (l, res)


@pytest.mark.parametrize("T,kind,seed", [(1, "gauss", 11), (5, "gauss", 22), (8, "clustered", 12)])
def test_nvfp4_stack_call_matches_oracle_every_layer(stack, T, kind, seed):
    """All 47 NVFP4 layers in one persistent launch (flint_moe_forward_layers),
    the same x for every layer: every layer against the oracle on the same
    NVFP4 codes."""
    layers, handles = stack
    xb = gen.x_gaussian(seed, T) if kind == "gauss" else gen.x_clustered(seed, T)[0]
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    ys = [torch.full_like(x, float("nan")) for _ in handles]
    flint.flint_moe_forward_layers(handles, [x] * N_LAYERS, T, ys)
    torch.cuda.synchronize()
    for l in range(N_LAYERS):
        y = ys[l].float().cpu().numpy()
        assert np.isfinite(y).all(), l
        ref, alt = nvfp4_oracle(*layers[l]).forward_with_alternatives(xb)
        res = compare(y, ref, alt)
        assert res["ok"], (l, res)


def test_nvfp4_stack_call_chained_and_graph_replay(stack):
    """Odd layers read the previous layer's output; the captured launch
    replays to the same bits as the direct call."""
    layers, handles = stack
    T = 4
    xb = gen.x_gaussian(33, T)
    x0 = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    ys = [torch.full_like(x0, float("nan")) for _ in range(N_LAYERS)]
    xs = [x0 if l % 2 == 0 else ys[l - 1] for l in range(N_LAYERS)]
    flint.flint_moe_forward_layers(handles, xs, T, ys)
    torch.cuda.synchronize()
    direct = [y.clone() for y in ys]
    for l in range(N_LAYERS):
        y = ys[l].float().cpu().numpy()
        assert np.isfinite(y).all(), l
        inp = xb if l % 2 == 0 else ys[l - 1].view(torch.int16).cpu().numpy().view(np.uint16)
        ref, alt = nvfp4_oracle(*layers[l]).forward_with_alternatives(inp)
        res = compare(y, ref, alt)
        assert res["ok"], (l, res)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        flint.flint_moe_forward_layers(handles, xs, T, ys, s)
    for _ in range(2):
        for y in ys:
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for l in range(N_LAYERS):
            assert torch.equal(ys[l], direct[l]), l
