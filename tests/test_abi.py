"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
symbol include/flint_moe.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import re

import pytest

from sparse_moe_transformer_03_b300 import build as flint_build
from sparse_moe_transformer_03_b300 import flint


@pytest.fixture(scope="module")
def lib():
    flint_build.build()
    return flint.load_library()


def test_exports_every_declared_symbol(lib):
    names = flint.declared_symbols()
    assert {"flint_moe_create", "flint_moe_forward", "flint_moe_route_only", "flint_moe_destroy"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_header_constants_match_binding():
    src = open(flint.HEADER).read()
    consts = dict(re.findall(r"#define (FLINT_\w+) (\d+)", src))
    assert int(consts["FLINT_HIDDEN"]) == flint.H
    assert int(consts["FLINT_INTER"]) == flint.I
    assert int(consts["FLINT_EXPERTS"]) == flint.E
    assert int(consts["FLINT_TOPK"]) == flint.TOPK
    assert int(consts["FLINT_CHUNK"]) == flint.CHUNK
    assert int(consts["FLINT_DECODE_MAX_T"]) == flint.DECODE_MAX_T
    assert int(consts["FLINT_STACK_MAX_T"]) == flint.STACK_MAX_T
    assert int(consts["FLINT_LM_HEAD_MAX_T"]) == flint.LM_HEAD_MAX_T
    assert int(consts["FLINT_STACK_MAX_LAYERS"]) == flint.STACK_MAX_LAYERS
    enums = dict(re.findall(r"(FLINT_(?:OK|ERR_\w+)) = (\d+)", src))
    assert {int(v): k for k, v in enums.items()} == flint.STATUS


def test_status_strings(lib):
    for code, name in flint.STATUS.items():
        assert flint.flint_status_string(code) == name


def test_host_argument_checks(lib):
    P = ctypes.c_void_p
    # null handle / null buffers / bad T: rejected before any CUDA call
    assert lib.flint_moe_forward(None, P(16), 1, P(4096 * 16), None) == 1
    assert lib.flint_moe_route_only(None, P(16), None, 1, P(32), P(64), None, None, None) == 1
    assert lib.flint_moe_destroy(None) == 0
    h = P()
    assert lib.flint_moe_create(ctypes.byref(h), None, None, None, None, None, 0) == 1
    arr = (P * 256)()
    sh = (P * 2)()
    assert lib.flint_moe_create(ctypes.byref(h), P(256), None, arr, arr, sh, 0) == 1  # null experts
    for i in range(256):
        arr[i] = 4096 * (i + 1)
    sh[0], sh[1] = 1 << 30, (1 << 30) + 4096
    assert lib.flint_moe_create(ctypes.byref(h), P(256), None, arr, arr, sh, 7) == 1  # bad dtype
    assert lib.flint_moe_create(ctypes.byref(h), P(258), None, arr, arr, sh, 0) == 1  # misaligned router
    arr[3] = 4096 * 4 + 8
    assert lib.flint_moe_create(ctypes.byref(h), P(256), None, arr, arr, sh, 0) == 1  # misaligned expert
    assert lib.flint_debug_bounded_wait(0, None) == 1
    # the stack call: null arrays, no layers, bad T, a null handle
    hs = (P * 2)()
    xs = (P * 2)(4096, 8192 * 4)
    ys = (P * 2)(4096 * 64, 4096 * 128)
    assert lib.flint_moe_forward_layers(None, 2, xs, 1, ys, None) == 1
    assert lib.flint_moe_forward_layers(hs, 0, xs, 1, ys, None) == 1
    assert lib.flint_moe_forward_layers(hs, 2, xs, 0, ys, None) == 1
    assert lib.flint_moe_forward_layers(hs, 2, None, 1, ys, None) == 1
    assert lib.flint_moe_forward_layers(hs, 2, xs, 1, ys, None) == 1      # null handles


def test_kernel_event_hook_rejects_bad_arguments():
    """Argument checks of the profiling hook run on the host (no GPU needed)."""
    from sparse_moe_transformer_03_b300 import flint
    lib = flint.load_library()
    assert lib.flint_moe_set_kernel_events(None, 1, None, None) == 1       # null handle


def test_nvfp4_create_rejects_null_parts():
    """NVFP4 entries with a null code or scale pointer are rejected before any device call."""
    import ctypes
    from sparse_moe_transformer_03_b300 import flint
    lib = flint.load_library()
    bad = flint.flint_nvfp4_t(None, None, 1.0)
    ok = flint.flint_nvfp4_t(16, 16, 1.0)       # non-null placeholders, never dereferenced on the device
    entries = (ctypes.c_void_p * 256)(*([ctypes.addressof(ok)] * 255 + [ctypes.addressof(bad)]))
    shared = (ctypes.c_void_p * 2)(ctypes.addressof(ok), ctypes.addressof(ok))
    h = ctypes.c_void_p()
    rc = lib.flint_moe_create(ctypes.byref(h), ctypes.c_void_p(16), None, entries, entries, shared, 1)
    assert rc == 1 and not h.value


def test_lm_head_host_argument_checks(lib):
    """The output layer's calls reject bad arguments before any CUDA call."""
    P = ctypes.c_void_p
    lib.flint_lm_head_create.argtypes = [ctypes.POINTER(P), ctypes.POINTER(flint.flint_nvfp4_t), ctypes.c_int]
    h = P()
    assert lib.flint_lm_head_create(None, None, 16) == 1
    assert lib.flint_lm_head_create(ctypes.byref(h), None, 16) == 1
    w = flint.flint_nvfp4_t(4096, 8192, 1.0)
    null_w = flint.flint_nvfp4_t(None, 8192, 1.0)
    assert lib.flint_lm_head_create(ctypes.byref(h), ctypes.byref(null_w), 16) == 1
    for V in (0, -16, 8, 24, 100):
        assert lib.flint_lm_head_create(ctypes.byref(h), ctypes.byref(w), V) == 1, V
    assert h.value is None
    lib.flint_lm_head_forward.argtypes = [P, P, ctypes.c_int, P, P]
    assert lib.flint_lm_head_forward(None, P(4096), 1, P(1 << 20), None) == 1
    assert lib.flint_lm_head_destroy(None) == 0
