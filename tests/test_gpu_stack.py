"""The 47-layer decode stack at full size, in the launch configuration the
benchmark times (every layer's forward captured into one CUDA graph and
replayed), with sampled layers checked against the fp64 oracle."""
import numpy as np
import pytest
import torch

from oracle.reference import LayerOracle, compare
from sparse_moe_transformer_03_b300 import flint
from synth import device, gen

pytestmark = pytest.mark.gpu

N_LAYERS = 47
SAMPLED = (0, 23, 46)


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


@pytest.mark.parametrize("T,kind,seed", [(1, "gauss", 11), (8, "clustered", 12)])
def test_stack_graph_replay_matches_oracle(stack, T, kind, seed):
    layers, handles = stack
    xb = gen.x_gaussian(seed, T) if kind == "gauss" else gen.x_clustered(seed, T)[0]
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    ys = [torch.full_like(x, float("nan")) for _ in range(N_LAYERS)]
    s = torch.cuda.Stream()

    def step():
        for l in range(N_LAYERS):
            flint.flint_moe_forward(handles[l], x, T, ys[l], s)

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
    for l in SAMPLED:
        y = ys[l].float().cpu().numpy()
        assert np.isfinite(y).all()
        ref, alt = LayerOracle.from_bf16_layer(layers[l]).forward_with_alternatives(xb)
        res = compare(y, ref, alt)
        assert res["ok"], (l, res)
