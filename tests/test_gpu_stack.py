"""The 47-layer decode stack at full size, in the launch configuration the
benchmark times (every layer's forward captured into one CUDA graph and
replayed), every layer checked against the fp64 oracle at T = 1, 8 and 32."""
import numpy as np
import pytest
import torch

from oracle.reference import LayerOracle, compare
from sparse_moe_transformer_03_b300 import flint
from synth import device, gen

pytestmark = pytest.mark.gpu

N_LAYERS = 47


@pytest.fixture(scope="module")
def stack():
    device.build()
    layers = [device.LayerWeights(1, l, True) for l in range(N_LAYERS)]
    handles = [flint.flint_moe_create(lw.router_W, lw.router_b, list(lw.gate_up[:256]), list(lw.down[:256]),
                                      (lw.gate_up[256], lw.down[256])) for lw in layers]
    yield layers, handles
    for h in handles:
        flint.flint_moe_destroy(h)
    del layers
    torch.cuda.empty_cache()


def replay_stack(handles, xb, T):
    """Capture the 47 forwards as one graph, poison the outputs, replay three
    times; returns the outputs of every layer."""
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    ys = [torch.full_like(x, float("nan")) for _ in handles]
    s = torch.cuda.Stream()

    def step():
        for l, h in enumerate(handles):
            flint.flint_moe_forward(h, x, T, ys[l], s)

    with torch.cuda.stream(s):
        step()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for y in ys:
        y.fill_(float("nan"))
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    return [y.float().cpu().numpy() for y in ys]


@pytest.mark.parametrize("T,kind,seed", [(1, "gauss", 11), (8, "clustered", 12), (32, "clustered", 13)])
def test_stack_graph_replay_matches_oracle(stack, T, kind, seed):
    layers, handles = stack
    xb = gen.x_gaussian(seed, T) if kind == "gauss" else gen.x_clustered(seed, T)[0]
    ys = replay_stack(handles, xb, T)
    for l in range(N_LAYERS):
        assert np.isfinite(ys[l]).all(), l
        ref, alt = LayerOracle.from_bf16_layer(layers[l]).forward_with_alternatives(xb)
        res = compare(ys[l], ref, alt)
        assert res["ok"], (l, res)
