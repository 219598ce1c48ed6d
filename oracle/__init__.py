"""Float64 CPU oracle of XAttention block-sparse chunked prefill.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference leg of ``bench.py``; never by the library.
"""
from .xattn_oracle import *  # noqa: F401,F403
from . import xattn_oracle  # noqa: F401
