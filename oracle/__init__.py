"""CPU oracle of the DeepSeek-V4 KV-cache write path (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``kvq_oracle.c`` (plain,
single-threaded C, no fused multiply-add) through ctypes and numpy; it imports
nothing from the CUDA library and the library imports nothing from it.
"""
from .oracle import *  # noqa: F401,F403
from .oracle import build, lib  # noqa: F401
