"""Flint mixture-of-experts FFN layer for B300 (sm_103a): CUDA kernels behind a C ABI.

The compute lives in ``libflint_moe.so`` (``csrc/``); :mod:`.flint` is its
ctypes binding.  See ``include/flint_moe.h`` for the contract.
"""
from . import flint  # noqa: F401
from .flint import (FLINT_BF16, FLINT_NVFP4, FlintError, flint_moe_create, flint_moe_destroy,  # noqa: F401
                    flint_moe_forward, flint_moe_route_only, flint_status_string)
