"""Shared fixtures of the GPU tests: device layers from the seeded generator."""
import numpy as np
import pytest
import torch

from synth import device, gen

_layers = {}


def layer(seed, layer_idx, with_bias):
    """Cached device layer (about 1.6 GB) generated on cuda:0."""
    key = (seed, layer_idx, with_bias)
    if key not in _layers:
        if len(_layers) >= 2:
            _layers.pop(next(iter(_layers)))
            torch.cuda.empty_cache()
        _layers[key] = device.LayerWeights(seed, layer_idx, with_bias)
    return _layers[key]


def to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def handle_for(lw):
    from sparse_moe_transformer_03_b300 import flint
    return flint.flint_moe_create(lw.router_W, lw.router_b, list(lw.gate_up[:256]), list(lw.down[:256]),
                                  (lw.gate_up[256], lw.down[256]))


def nvfp4_oracle(lw, q):
    """fp64 oracle layer on the exactly decoded NVFP4 weights of `q`
    (device.LayerNVFP4 of `lw`); the router stays bf16."""
    import oracle
    from oracle.reference import LayerOracle

    def mats(e):
        (pg, sg, tg), (pd, sd, td) = q.expert_parts(e)
        return (oracle.Mat(packed=pg, scales=sg, tensor_scale=tg), oracle.Mat(packed=pd, scales=sd, tensor_scale=td))
    return LayerOracle(lw.router_bits(), lw.bias_host(), mats, mats(lw.E), lw.E)


def x_for(kind, seed, T):
    if kind == "gauss":
        return gen.x_gaussian(seed, T)
    return gen.x_clustered(seed, T)[0]
