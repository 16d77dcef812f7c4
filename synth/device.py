"""Device-side input generation (CUDA, ``csrc/synth_gen.cu``) for large weight stacks.

Draws exactly the streams of :mod:`synth.gen` (same keys, same Box-Muller
normals in double precision, same rounding to bf16), directly into torch
CUDA tensors.  Input generation only.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

from . import gen

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csrc", "synth_gen.cu")
_LIB = os.path.join(_HERE, "libflint_synth.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        nvcc = "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc"
        subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                               "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                               "-o", _LIB + ".tmp", _SRC])
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB):
            raise RuntimeError(f"synth CUDA generator not built ({_LIB}); run __graft_entry__.build()")
        lib = ctypes.CDLL(_LIB)
        lib.synth_fill_normal_bf16.restype = ctypes.c_int
        lib.synth_fill_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32,
                                               ctypes.c_uint32, ctypes.c_uint32, ctypes.c_double, ctypes.c_void_p]
        lib.synth_fill_normal_bf16_batched.restype = ctypes.c_int
        lib.synth_fill_normal_bf16_batched.argtypes = [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64,
                                                       ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                                       ctypes.c_uint32, ctypes.c_double, ctypes.c_void_p]
        lib.synth_fill_normal_f32.restype = ctypes.c_int
        lib.synth_fill_normal_f32.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                              ctypes.c_uint32, ctypes.c_double, ctypes.c_void_p]
        lib.synth_nvfp4_quantize.restype = ctypes.c_int
        lib.synth_nvfp4_quantize.argtypes = [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p]
        _lib = lib
    return _lib


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def fill_normal_bf16(t, seed: int, layer: int, tensor: int, std: float, start: int = 0, stream=None):
    """Fill a contiguous bf16 CUDA tensor with std * N(0,1) of a stream."""
    import torch
    assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
    rc = _load().synth_fill_normal_bf16(ctypes.c_void_p(t.data_ptr()), t.numel(), start, seed, layer, tensor,
                                        float(std), _stream_ptr(stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_normal_bf16 failed ({rc})")
    return t


def fill_normal_bf16_batched(t, seed: int, layer: int, tensor0: int, tensor_stride: int, std: float,
                             stream=None):
    """Fill t[i] (t of shape [n, ...], contiguous bf16) with stream
    (seed, layer, tensor0 + i * tensor_stride) for every i."""
    import torch
    assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
    n = t.shape[0]
    rc = _load().synth_fill_normal_bf16_batched(ctypes.c_void_p(t.data_ptr()), n, t.numel() // n, seed, layer,
                                                tensor0, tensor_stride, float(std), _stream_ptr(stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_normal_bf16_batched failed ({rc})")
    return t


def fill_normal_f32(t, seed: int, layer: int, tensor: int, std: float, stream=None):
    import torch
    assert t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()
    rc = _load().synth_fill_normal_f32(ctypes.c_void_p(t.data_ptr()), t.numel(), seed, layer, tensor, float(std),
                                       _stream_ptr(stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_normal_f32 failed ({rc})")
    return t


class LayerWeights:
    """One MoE layer's weights in device memory, generated from (seed, layer).

    gate_up: bf16 [257][2I][H] (index 256 = shared expert), down: bf16
    [257][H][I], router_W: bf16 [E][H], router_b: fp32 [E] or None."""

    def __init__(self, seed: int, layer: int, with_bias: bool, device="cuda",
                 E: int = gen.E, H: int = gen.H, I: int = gen.I):
        import torch
        self.seed, self.layer, self.E, self.H, self.I = seed, layer, E, H, I
        self.router_W = torch.empty((E, H), dtype=torch.bfloat16, device=device)
        fill_normal_bf16(self.router_W, seed, layer, gen.T_ROUTER_W, 1.0 / (H ** 0.5))
        self.router_b = None
        if with_bias:
            self.router_b = torch.empty((E,), dtype=torch.float32, device=device)
            fill_normal_f32(self.router_b, seed, layer, gen.T_ROUTER_B, gen.BIAS_STD)
        self.gate_up = torch.empty((E + 1, 2 * I, H), dtype=torch.bfloat16, device=device)
        self.down = torch.empty((E + 1, H, I), dtype=torch.bfloat16, device=device)
        fill_normal_bf16_batched(self.gate_up, seed, layer, gen.gate_up_tensor(0), 2, gen.WEIGHT_STD)
        fill_normal_bf16_batched(self.down, seed, layer, gen.down_tensor(0), 2, gen.WEIGHT_STD)

    def expert_bits(self, e: int):
        """(gate_up, down) of expert e as numpy uint16 bf16 bits (host copies)."""
        import torch
        gu = self.gate_up[e].view(torch.int16).cpu().numpy().view("uint16")
        dn = self.down[e].view(torch.int16).cpu().numpy().view("uint16")
        return gu, dn

    def router_bits(self):
        import torch
        return self.router_W.view(torch.int16).cpu().numpy().view("uint16")

    def bias_host(self):
        return None if self.router_b is None else self.router_b.cpu().numpy()


def nvfp4_quantize(w, stream=None):
    """NVFP4 encoding (as synth.gen.nvfp4_quantize) of a bf16 CUDA tensor
    [n][R][K] (or [R][K]): returns (packed uint8 [n][R][K/2], scales uint8
    [n][R][K/16], tensor scales float32 [n]) as CUDA tensors."""
    import torch
    assert w.is_cuda and w.dtype == torch.bfloat16 and w.is_contiguous()
    w3 = w if w.dim() == 3 else w.unsqueeze(0)
    n, R, K = w3.shape
    packed = torch.empty((n, R, K // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((n, R, K // 16), dtype=torch.uint8, device=w.device)
    ts = torch.empty((n,), dtype=torch.float32, device=w.device)
    scratch = torch.empty((n,), dtype=torch.int32, device=w.device)
    rc = _load().synth_nvfp4_quantize(ctypes.c_void_p(w3.data_ptr()), n, R, K, ctypes.c_void_p(packed.data_ptr()),
                                      ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(ts.data_ptr()),
                                      ctypes.c_void_p(scratch.data_ptr()), _stream_ptr(stream))
    if rc != 0:
        raise RuntimeError(f"synth_nvfp4_quantize failed ({rc})")
    return packed, scales, ts


class LayerNVFP4:
    """A layer's expert weights in NVFP4, quantised on the device from a
    bf16 layer (synth.device.LayerWeights); the router stays bf16 (borrowed
    from the bf16 layer, which must stay alive while this object is used
    for the router)."""

    def __init__(self, lw):
        self.E = lw.E
        self.router_W, self.router_b = lw.router_W, lw.router_b
        self._router_bits, self._bias = None, None
        self.gu = nvfp4_quantize(lw.gate_up)     # ([257][1024][1024], [257][1024][128], [257])
        self.dn = nvfp4_quantize(lw.down)        # ([257][2048][256], [257][2048][32], [257])
        self.ts_gu = self.gu[2].cpu().numpy()
        self.ts_dn = self.dn[2].cpu().numpy()

    def create_args(self):
        """(gate_up entries, down entries, shared entries) for flint_moe_create(dtype=FLINT_NVFP4)."""
        gu = [(self.gu[0][e], self.gu[1][e], float(self.ts_gu[e])) for e in range(self.E + 1)]
        dn = [(self.dn[0][e], self.dn[1][e], float(self.ts_dn[e])) for e in range(self.E + 1)]
        return gu[:self.E], dn[:self.E], (gu[self.E], dn[self.E])

    def expert_parts(self, e: int):
        """Host copies ((packed, scales, ts) of gate_up, same of down) of expert e."""
        return ((self.gu[0][e].cpu().numpy(), self.gu[1][e].cpu().numpy(), self.ts_gu[e]),
                (self.dn[0][e].cpu().numpy(), self.dn[1][e].cpu().numpy(), self.ts_dn[e]))
