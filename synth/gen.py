"""Seeded synthetic inputs for the Flint MoE layer (host side, numpy).

This module only makes inputs: random tensors with the shapes and value
distributions of the workloads, and the NVFP4 encoding of given weights.  It
holds none of the layer's arithmetic (no router, top-k, SwiGLU or combine).
The CUDA generator in ``csrc/synth_gen.cu`` draws the very same numbers, so
large weight stacks can be produced directly in device memory.

Counter-based generator
-----------------------
Each tensor is a stream keyed by (seed, layer, tensor id).  The key is the
SplitMix64 finaliser (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) applied to ``seed<<32 | layer<<16 | tensor``;
draw i of a stream is that finaliser applied to ``key + (i+1)*0x9E3779B97F4A7C15``
(mod 2^64), i.e. SplitMix64's i-th output.  A uniform is
``((r >> 11) + 0.5) * 2^-53`` (never 0 or 1).  Normal deviates come from the
Box-Muller transform in double precision: pair p uses draws 2p and 2p+1,
``rad = sqrt(-2 ln u1)``, ``theta = 2*pi*u2``; element 2p is ``rad*cos(theta)``
and element 2p+1 is ``rad*sin(theta)``.  A bf16 tensor stores
``bf16_rne(float32_rn(std * z))``.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids of the streams
T_X = 1
T_CENTROID0 = 2          # 2..5: the four cluster centroids
T_CLUSTER = 6            # cluster id per token
T_ROUTER_W = 10
T_ROUTER_B = 11
T_LM_HEAD = 20           # output layer (lm_head) [V][H]
T_GATE_UP0 = 100         # gate_up of expert e: 100 + 2e  (e = 256 is the shared expert)
T_DOWN0 = 101            # down    of expert e: 101 + 2e

H = 2048
I = 512
E = 256
K_TOP = 6
SHARED = 256             # expert index used for the shared expert's streams

WEIGHT_STD = 0.02
ROUTER_STD = 1.0 / np.sqrt(2048.0)
BIAS_STD = 0.5


def gate_up_tensor(e: int) -> int:
    return T_GATE_UP0 + 2 * e


def down_tensor(e: int) -> int:
    return T_DOWN0 + 2 * e


def _mix64(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def stream_key(seed: int, layer: int, tensor: int) -> np.uint64:
    assert 0 <= seed < 2**32 and 0 <= layer < 2**16 and 0 <= tensor < 2**16
    base = np.array([(seed << 32) | (layer << 16) | tensor], dtype=np.uint64)
    return _mix64(base)[0]


def draws(seed: int, layer: int, tensor: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit draws start..start+count-1 of the stream."""
    key = stream_key(seed, layer, tensor)
    i = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = key + (i + np.uint64(1)) * GOLDEN
    return _mix64(z)


def uniforms(seed, layer, tensor, start, count) -> np.ndarray:
    r = draws(seed, layer, tensor, start, count)
    return ((r >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normals(seed: int, layer: int, tensor: int, count: int, start: int = 0) -> np.ndarray:
    """Standard normal deviates start..start+count-1 of a stream (float64)."""
    p0 = start // 2
    p1 = (start + count + 1) // 2
    u = uniforms(seed, layer, tensor, 2 * p0, 2 * (p1 - p0))
    u1 = u[0::2]
    u2 = u[1::2]
    rad = np.sqrt(-2.0 * np.log(u1))
    theta = (2.0 * np.pi) * u2
    z = np.empty(2 * (p1 - p0), dtype=np.float64)
    z[0::2] = rad * np.cos(theta)
    z[1::2] = rad * np.sin(theta)
    off = start - 2 * p0
    return z[off:off + count]


# --------------------------------------------------------------------------
# number formats (encoding only)
# --------------------------------------------------------------------------

def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); finite inputs."""
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_bf16_bits(values: np.ndarray) -> np.ndarray:
    """float64 -> float32 (round to nearest) -> bf16 bits (ties to even)."""
    return f32_to_bf16_bits(np.asarray(values, dtype=np.float64).astype(np.float32))


def normal_bf16(seed, layer, tensor, shape, std, start=0) -> np.ndarray:
    n = int(np.prod(shape))
    z = normals(seed, layer, tensor, n, start)
    return to_bf16_bits(std * z).reshape(shape)


# --------------------------------------------------------------------------
# the workloads' inputs
# --------------------------------------------------------------------------

def rms_normalise(v: np.ndarray) -> np.ndarray:
    """Rows scaled to unit root-mean-square (no epsilon, no gain)."""
    v = np.asarray(v, dtype=np.float64)
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True))


def x_gaussian(seed: int, T: int, H_: int = H) -> np.ndarray:
    """x ~ N(0, 1) per element, each token RMS-normalised; bf16 bits [T][H]."""
    z = normals(seed, 0, T_X, T * H_).reshape(T, H_)
    return to_bf16_bits(rms_normalise(z))


def x_clustered(seed: int, T: int, H_: int = H, n_clusters: int = 4, sigma: float = 0.3):
    """Tokens from a Gaussian mixture: centroids c_k ~ N(0, I) rescaled to unit
    RMS, a uniform cluster id per token, x = c_id + sigma * eps, then each token
    RMS-normalised.  Returns (bf16 bits [T][H], cluster ids [T])."""
    cents = np.stack([rms_normalise(normals(seed, 0, T_CENTROID0 + c, H_)) for c in range(n_clusters)])
    cid = (draws(seed, 0, T_CLUSTER, 0, T) % np.uint64(n_clusters)).astype(np.int64)
    eps = normals(seed, 0, T_X, T * H_).reshape(T, H_)
    x = cents[cid] + sigma * eps
    return to_bf16_bits(rms_normalise(x)), cid


def router_weight(seed: int, layer: int, E_: int = E, H_: int = H) -> np.ndarray:
    return normal_bf16(seed, layer, T_ROUTER_W, (E_, H_), 1.0 / np.sqrt(H_))


def router_bias(seed: int, layer: int, E_: int = E) -> np.ndarray:
    z = normals(seed, layer, T_ROUTER_B, E_)
    return (BIAS_STD * z).astype(np.float32)


def expert_gate_up(seed: int, layer: int, e: int, H_: int = H, I_: int = I) -> np.ndarray:
    return normal_bf16(seed, layer, gate_up_tensor(e), (2 * I_, H_), WEIGHT_STD)


def expert_down(seed: int, layer: int, e: int, H_: int = H, I_: int = I) -> np.ndarray:
    return normal_bf16(seed, layer, down_tensor(e), (H_, I_), WEIGHT_STD)


# --------------------------------------------------------------------------
# NVFP4 encoding of a bf16 matrix
# --------------------------------------------------------------------------
# Per matrix: s_t = amax / (6 * 448) in fp32 (1 if amax == 0).  Per block of
# 16 consecutive columns: s_b = e4m3_rn_satfinite(amax_b / (6 * s_t)); each
# element q = e2m1_rn(w / (dec(s_b) * s_t)) (ties to even, clamped to +-6),
# or 0 where the block scale decodes to zero.  Packed two per byte, the even
# column in the low nibble; scales laid out [rows][cols/16].

def e4m3_encode_rn_sat(v: np.ndarray) -> np.ndarray:
    """Non-negative float32 -> E4M3 code, round to nearest (ties to even),
    saturating at 448 (code 0x7E)."""
    v = np.asarray(v, dtype=np.float64)   # exact widening of the float32 value
    assert np.all(v >= 0)
    out = np.zeros(v.shape, dtype=np.uint8)
    nz = v > 0
    mant, ex = np.frexp(v[nz])            # v = mant * 2^ex, mant in [0.5, 1)
    ue = ex - 1                           # unbiased exponent of the leading bit
    step_exp = np.where(ue < -6, -9, ue - 3)
    q = np.rint(np.ldexp(v[nz], -step_exp))   # exact scaling, ties to even
    sub = ue < -6
    code = np.where(sub, q, 0).astype(np.int64)
    m = q - 8
    e = ue + 7
    carry = q >= 16
    e = np.where(carry, e + 1, e)
    m = np.where(carry, 0, m)
    code = np.where(sub, code, (e.astype(np.int64) << 3) | m.astype(np.int64))
    code = np.minimum(code, 0x7E)
    out[nz] = code.astype(np.uint8)
    return out


def e4m3_code_to_f32(code: np.ndarray) -> np.ndarray:
    c = np.asarray(code, dtype=np.int64)
    e = (c >> 3) & 15
    m = c & 7
    v = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    v = np.where((c >> 7) & 1, -v, v)
    return v.astype(np.float32)


def e2m1_encode_rn(v: np.ndarray) -> np.ndarray:
    """float32 -> E2M1 code (magnitude index into 0,.5,1,1.5,2,3,4,6),
    round to nearest with ties to even, clamped at 6."""
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v)
    i = np.full(v.shape, 7, dtype=np.uint8)
    i = np.where(a <= 5.0, 6, i)
    i = np.where(a < 3.5, 5, i)
    i = np.where(a <= 2.5, 4, i)
    i = np.where(a < 1.75, 3, i)
    i = np.where(a <= 1.25, 2, i)
    i = np.where(a < 0.75, 1, i)
    i = np.where(a <= 0.25, 0, i).astype(np.uint8)
    neg = (v < 0) & (i > 0)
    return (i | np.where(neg, 8, 0)).astype(np.uint8)


def nvfp4_quantize(bits: np.ndarray):
    """bf16 bits [R][K] -> (packed uint8 [R][K/2], scales uint8 [R][K/16], tensor_scale fp32)."""
    w = bf16_bits_to_f32(bits).astype(np.float32)
    R, K = w.shape
    assert K % 16 == 0
    amax = np.float32(np.max(np.abs(w))) if w.size else np.float32(0)
    if amax == 0:
        s_t = np.float32(1.0)
    else:
        s_t = np.float32(amax / np.float32(6.0 * 448.0))
    blocks = w.reshape(R, K // 16, 16)
    amax_b = np.max(np.abs(blocks), axis=2).astype(np.float32)
    denom = np.float32(np.float32(6.0) * s_t)
    sb = e4m3_encode_rn_sat((amax_b / denom).astype(np.float32))
    sdec = e4m3_code_to_f32(sb)
    scale = (sdec * s_t).astype(np.float32)                     # [R][K/16]
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    qv = (blocks / safe[:, :, None]).astype(np.float32)
    q = e2m1_encode_rn(qv)
    q = np.where(scale[:, :, None] > 0, q, 0).astype(np.uint8).reshape(R, K)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return packed, sb.astype(np.uint8), np.float32(s_t)
