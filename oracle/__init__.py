"""The fp64 CPU oracle of the Flint MoE FFN layer -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
binding) never does.
"""
from .oracle import *  # noqa: F401,F403
