"""ctypes binding of the fp64 CPU oracle (``flint_oracle.c``) -- test infrastructure only.

Functions take numpy arrays: bf16 tensors are passed as their uint16 bit
patterns, NVFP4 matrices as (packed uint8 [R][K/2], scales uint8 [R][K/16],
fp32 tensor scale).  Every computation happens in the C file in IEEE double.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "flint_oracle.c")
_LIB = os.path.join(_HERE, "libflint_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-o", _LIB + ".tmp", _SRC, "-lm", "-lpthread"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


class OracleMat(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32),
        ("rows", ctypes.c_int32),
        ("cols", ctypes.c_int32),
        ("bf16", ctypes.c_void_p),
        ("packed", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("tensor_scale", ctypes.c_float),
        ("pad_", ctypes.c_int32),
    ]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_e2m1_decode.restype = ctypes.c_double
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_sigmoid.restype = ctypes.c_double
        lib.oracle_sigmoid.argtypes = [ctypes.c_double]
        lib.oracle_silu.restype = ctypes.c_double
        lib.oracle_silu.argtypes = [ctypes.c_double]
        lib.oracle_nvfp4_dequant.restype = None
        lib.oracle_nvfp4_dequant.argtypes = [i, i, P, P, ctypes.c_float, P]
        lib.oracle_router_logits.restype = None
        lib.oracle_router_logits.argtypes = [i, i, i, P, P, P, P]
        lib.oracle_select.restype = None
        lib.oracle_select.argtypes = [i, i, i, P, P, P]
        lib.oracle_expert.restype = None
        lib.oracle_expert.argtypes = [i, i, P, P, P, P]
        lib.oracle_moe_forward.restype = ctypes.c_int
        lib.oracle_moe_forward.argtypes = [i, i, i, i, i, P, P, P, P, P, P, P, P, P, P, P, P, i]
        lib.oracle_permutation.restype = None
        lib.oracle_permutation.argtypes = [i, i, i, P, P, P]
        lib.oracle_lm_head.argtypes = [i, i, P, ctypes.POINTER(OracleMat), i, P, P]
        lib.oracle_lm_head.restype = None
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


# --------------------------------------------------------------------------
# weight matrices
# --------------------------------------------------------------------------

class Mat:
    """A weight matrix handed to the oracle: bf16 bits or NVFP4 parts.

    Keeps references to its numpy buffers so the C struct stays valid."""

    def __init__(self, bf16=None, packed=None, scales=None, tensor_scale=None, rows=None, cols=None):
        self._keep = []
        if bf16 is not None:
            b = _u16(bf16)
            self._keep.append(b)
            self.s = OracleMat(0, b.shape[0], b.shape[1], b.ctypes.data, None, None, 0.0, 0)
        elif packed is not None:
            pk = np.ascontiguousarray(packed, dtype=np.uint8)
            sc = np.ascontiguousarray(scales, dtype=np.uint8)
            r, kh = pk.shape
            assert sc.shape == (r, kh * 2 // 16), (sc.shape, pk.shape)
            self._keep += [pk, sc]
            self.s = OracleMat(1, r, kh * 2, None, pk.ctypes.data, sc.ctypes.data,
                               float(np.float32(tensor_scale)), 0)
        else:
            self.s = OracleMat(-1, rows or 0, cols or 0, None, None, None, 0.0, 0)

    @staticmethod
    def absent():
        return Mat()


def _mat_array(mats):
    arr = (OracleMat * len(mats))()
    for i, m in enumerate(mats):
        arr[i] = m.s
    return arr


# --------------------------------------------------------------------------
# scalar helpers
# --------------------------------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))


def e2m1_decode(code: int) -> float:
    return _load().oracle_e2m1_decode(int(code))


def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(int(code))


def sigmoid(z: float) -> float:
    return _load().oracle_sigmoid(float(z))


def silu(z: float) -> float:
    return _load().oracle_silu(float(z))


def nvfp4_dequant(packed, scales, tensor_scale) -> np.ndarray:
    pk = np.ascontiguousarray(packed, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.uint8)
    r, kh = pk.shape
    out = np.empty((r, kh * 2), dtype=np.float64)
    _load().oracle_nvfp4_dequant(r, kh * 2, _p(pk), _p(sc), float(np.float32(tensor_scale)), _p(out))
    return out


# --------------------------------------------------------------------------
# router / selection / experts / layer
# --------------------------------------------------------------------------

def router_logits(x_bits, Wr_bits, bias=None) -> np.ndarray:
    x = _u16(x_bits)
    W = _u16(Wr_bits)
    T, H = x.shape
    E = W.shape[0]
    assert W.shape[1] == H
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.empty((T, E), dtype=np.float64)
    _load().oracle_router_logits(T, E, H, _p(x), _p(W), _p(b), _p(out))
    return out


def select(logits, k: int = 6):
    l = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = l.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    _load().oracle_select(T, E, k, _p(l), _p(idx), _p(w))
    return idx, w


def expert(gate_up: Mat, down: Mat, x) -> np.ndarray:
    xr = np.ascontiguousarray(x, dtype=np.float64)
    H = xr.shape[0]
    I = gate_up.s.rows // 2
    o = np.empty(H, dtype=np.float64)
    g = OracleMat.from_buffer_copy(gate_up.s)
    d = OracleMat.from_buffer_copy(down.s)
    _load().oracle_expert(H, I, ctypes.byref(g), ctypes.byref(d), _p(xr), _p(o))
    return o


def moe_forward(x_bits, Wr_bits, bias, gate_up, down, shared, k: int = 6,
                idx_in=None, nthreads: int | None = None):
    """Evaluate the layer.

    gate_up/down: lists of ``Mat`` (length E; ``Mat.absent()`` for experts the
    caller knows are never selected).  shared: (gate_up Mat, down Mat) or None.
    Returns dict(y, logits, idx, w) with y in float64 [T][H]."""
    x = _u16(x_bits)
    W = _u16(Wr_bits)
    T, H = x.shape
    E = W.shape[0]
    assert len(gate_up) == E and len(down) == E
    I = None
    for m in gate_up:
        if m.s.kind >= 0:
            I = m.s.rows // 2
            break
    if I is None and shared is not None:
        I = shared[0].s.rows // 2
    if I is None:
        I = 1
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    gu = _mat_array(gate_up)
    dn = _mat_array(down)
    if shared is not None:
        sg = OracleMat.from_buffer_copy(shared[0].s)
        sd = OracleMat.from_buffer_copy(shared[1].s)
        sgp, sdp = ctypes.byref(sg), ctypes.byref(sd)
    else:
        sgp = sdp = None
    ii = None if idx_in is None else np.ascontiguousarray(idx_in, dtype=np.int32)
    y = np.empty((T, H), dtype=np.float64)
    logits = np.empty((T, E), dtype=np.float64)
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _load().oracle_moe_forward(T, E, H, I, k, _p(x), _p(W), _p(b), gu, dn, sgp, sdp,
                                    _p(ii), _p(y), _p(logits), _p(idx), _p(w), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: a selected expert has no weights supplied")
    return {"y": y, "logits": logits, "idx": idx, "w": w}


def lm_head(x_bits, W: Mat, rows=None) -> np.ndarray:
    """Output-layer logits [T][len(rows)] (every row of W when rows is None)
    of x (bf16 bits [T][H]) against W ([V][H], bf16 or NVFP4)."""
    x = _u16(x_bits)
    T, H = x.shape
    assert W.s.cols == H
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n = W.s.rows if r is None else len(r)
    if r is not None:
        assert ((r >= 0) & (r < W.s.rows)).all()
    out = np.empty((T, n), dtype=np.float64)
    _load().oracle_lm_head(T, H, _p(x), ctypes.byref(W.s), n, _p(r), _p(out))
    return out


def permutation(idx, E: int = 256):
    i = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = i.shape
    offsets = np.empty(E + 1, dtype=np.int32)
    gather = np.empty(T * k, dtype=np.int32)
    _load().oracle_permutation(T, E, k, _p(i), _p(offsets), _p(gather))
    return offsets, gather


__all__ = ["build", "Mat", "OracleMat", "bf16_to_double", "e2m1_decode", "e4m3_decode",
           "sigmoid", "silu", "nvfp4_dequant", "router_logits", "select", "expert",
           "moe_forward", "permutation", "lm_head"]
