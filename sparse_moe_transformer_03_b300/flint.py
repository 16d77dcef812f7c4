"""Thin ctypes binding of ``libflint_moe.so`` (C ABI in include/flint_moe.h).

Argument marshalling only: every step of the layer runs in the CUDA library.
The functions keep the C names.  Device buffers are passed as torch CUDA
tensors (or raw integer device addresses); streams as torch.cuda.Stream (or
None for the current stream).  There is no fallback: if the library is
missing this module raises on import of the library.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libflint_moe.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "flint_moe.h")

FLINT_BF16 = 0
FLINT_NVFP4 = 1

STATUS = {
    0: "FLINT_OK",
    1: "FLINT_ERR_INVALID_ARG",
    2: "FLINT_ERR_CUDA",
    3: "FLINT_ERR_OOM",
    4: "FLINT_ERR_DEVICE_TIMEOUT",
    5: "FLINT_ERR_DEVICE_BADINDEX",
    6: "FLINT_ERR_UNSUPPORTED",
    7: "FLINT_ERR_INTERNAL",
}

H, I, E, TOPK, CHUNK, DECODE_MAX_T = 2048, 512, 256, 6, 8192, 32
STACK_MAX_T, STACK_MAX_LAYERS = 8, 64
LM_HEAD_MAX_T = 32               # FLINT_LM_HEAD_MAX_T


class FlintError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


class flint_nvfp4_t(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("block_scales", ctypes.c_void_p), ("tensor_scale", ctypes.c_float)]


_lib = None


def load_library():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m sparse_moe_transformer_03_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32 = ctypes.c_void_p, ctypes.c_int
    lib.flint_moe_create.restype = I32
    lib.flint_moe_create.argtypes = [ctypes.POINTER(P), P, P, P, P, P, I32]
    lib.flint_moe_forward.restype = I32
    lib.flint_moe_forward.argtypes = [P, P, I32, P, P]
    lib.flint_moe_forward_layers.restype = I32
    lib.flint_moe_forward_layers.argtypes = [P, I32, P, I32, P, P]
    lib.flint_moe_route_only.restype = I32
    lib.flint_moe_route_only.argtypes = [P, P, P, I32, P, P, P, P, P]
    lib.flint_moe_destroy.restype = I32
    lib.flint_moe_destroy.argtypes = [P]
    lib.flint_status_string.restype = ctypes.c_char_p
    lib.flint_status_string.argtypes = [I32]
    lib.flint_moe_set_kernel_events.restype = I32
    lib.flint_moe_set_kernel_events.argtypes = [P, I32, P, P]
    lib.flint_permute_static.restype = I32
    lib.flint_permute_static.argtypes = [P, I32, P, P, P]
    lib.flint_debug_bounded_wait.restype = I32
    lib.flint_debug_bounded_wait.argtypes = [ctypes.c_uint64, P]
    lib.flint_lm_head_create.restype = I32
    lib.flint_lm_head_create.argtypes = [ctypes.POINTER(P), ctypes.POINTER(flint_nvfp4_t), I32]
    lib.flint_lm_head_forward.restype = I32
    lib.flint_lm_head_forward.argtypes = [P, P, I32, P, P]
    lib.flint_lm_head_destroy.restype = I32
    lib.flint_lm_head_destroy.argtypes = [P]
    _lib = lib
    return lib


def declared_symbols():
    """Names of the functions include/flint_moe.h declares."""
    src = open(HEADER).read()
    return re.findall(r"FLINT_API\s+[\w\s\*]+?\b(flint_\w+)\s*\(", src)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return ctypes.c_void_p(x)
    return ctypes.c_void_p(x.data_ptr())


def _stream(s):
    if s is None:
        import torch
        s = torch.cuda.current_stream()
    if isinstance(s, int):
        return ctypes.c_void_p(s)
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, rc):
    if rc != 0:
        raise FlintError(fn, rc)


def _ptr_array(ptrs):
    arr = (ctypes.c_void_p * len(ptrs))()
    for i, p in enumerate(ptrs):
        arr[i] = p if isinstance(p, int) else (p.data_ptr() if hasattr(p, "data_ptr") else ctypes.addressof(p))
    return arr


def flint_moe_create(router_W, router_b, gate_up, down, shared, dtype=FLINT_BF16):
    """Create a layer handle.

    router_W: bf16 [256][2048] tensor; router_b: fp32 [256] tensor or None.
    gate_up/down: 256 per-expert entries; shared: (gate_up, down).
    BF16: entries are bf16 CUDA tensors (or device addresses).
    NVFP4: entries are (packed, block_scales, tensor_scale) tuples of CUDA
    uint8 tensors and a float.  Returns the handle (an int)."""
    lib = load_library()
    keep = []

    def entry(v):
        if dtype == FLINT_NVFP4:
            pk, sc, ts = v
            st = flint_nvfp4_t(_ptr(pk).value, _ptr(sc).value, float(ts))
            keep.append(st)
            return ctypes.addressof(st)
        return v if isinstance(v, int) else v.data_ptr()

    gu = _ptr_array([entry(v) for v in gate_up])
    dn = _ptr_array([entry(v) for v in down])
    sh = _ptr_array([entry(shared[0]), entry(shared[1])])
    h = ctypes.c_void_p()
    rc = lib.flint_moe_create(ctypes.byref(h), _ptr(router_W), _ptr(router_b), gu, dn, sh, int(dtype))
    _check("flint_moe_create", rc)
    return h.value


def flint_moe_forward(h, x, T, y, stream=None):
    _check("flint_moe_forward", load_library().flint_moe_forward(ctypes.c_void_p(h), _ptr(x), int(T), _ptr(y),
                                                                 _stream(stream)))


def flint_moe_forward_layers(handles, xs, T, ys, stream=None):
    """n layers in order: ys[l] = layer handles[l] applied to xs[l] (device
    buffers bf16 [T][2048]; xs[l + 1] may be ys[l])."""
    n = len(handles)
    if len(xs) != n or len(ys) != n:
        raise ValueError("one x and one y per layer")
    hs = (ctypes.c_void_p * n)(*[int(h) for h in handles])
    xa = (ctypes.c_void_p * n)(*[_ptr(x).value for x in xs])
    ya = (ctypes.c_void_p * n)(*[_ptr(y).value for y in ys])
    _check("flint_moe_forward_layers",
           load_library().flint_moe_forward_layers(hs, n, xa, int(T), ya, _stream(stream)))


def flint_moe_route_only(h, x, logits, T, idx, w, offsets=None, gather_idx=None, stream=None):
    _check("flint_moe_route_only",
           load_library().flint_moe_route_only(ctypes.c_void_p(h), _ptr(x), _ptr(logits), int(T), _ptr(idx), _ptr(w),
                                               _ptr(offsets), _ptr(gather_idx), _stream(stream)))


FLINT_KERNEL_ROUTER, FLINT_KERNEL_GATE_UP, FLINT_KERNEL_DOWN, FLINT_KERNEL_COMBINE = 0, 1, 2, 3


def flint_moe_set_kernel_events(h, kernel, start=None, stop=None):
    """start/stop: torch.cuda.Event(enable_timing=True) (or raw cudaEvent_t), None to clear."""
    def ev(e):
        if e is None:
            return None
        if hasattr(e, "cuda_event"):
            if not e.cuda_event:
                e.record()        # torch creates the CUDA event on its first record
            return ctypes.c_void_p(e.cuda_event)
        return ctypes.c_void_p(int(e))
    _check("flint_moe_set_kernel_events",
           load_library().flint_moe_set_kernel_events(ctypes.c_void_p(h), int(kernel), ev(start), ev(stop)))


def flint_permute_static(idx, T, offsets, gather_idx, stream=None):
    _check("flint_permute_static",
           load_library().flint_permute_static(_ptr(idx), int(T), _ptr(offsets), _ptr(gather_idx), _stream(stream)))


def flint_moe_destroy(h):
    _check("flint_moe_destroy", load_library().flint_moe_destroy(ctypes.c_void_p(h) if h else None))


def flint_status_string(code):
    return load_library().flint_status_string(int(code)).decode()


def flint_lm_head_create(W, V):
    """Output-layer handle from W = (packed uint8 [V][1024], block_scales
    uint8 [V][128], tensor_scale) with CUDA tensors (or device addresses)."""
    pk, sc, ts = W
    st = flint_nvfp4_t(_ptr(pk).value, _ptr(sc).value, float(ts))
    h = ctypes.c_void_p()
    _check("flint_lm_head_create", load_library().flint_lm_head_create(ctypes.byref(h), ctypes.byref(st), int(V)))
    return h.value


def flint_lm_head_forward(h, x, T, logits, stream=None):
    _check("flint_lm_head_forward",
           load_library().flint_lm_head_forward(ctypes.c_void_p(h), _ptr(x), int(T), _ptr(logits), _stream(stream)))


def flint_lm_head_destroy(h):
    _check("flint_lm_head_destroy", load_library().flint_lm_head_destroy(ctypes.c_void_p(h) if h else None))


def flint_debug_bounded_wait(timeout_ns, stream=None):
    """Returns the raw status code (FLINT_ERR_DEVICE_TIMEOUT = 4 is the designed outcome)."""
    return load_library().flint_debug_bounded_wait(int(timeout_ns), _stream(stream))
