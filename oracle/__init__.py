"""CPU oracle for the 8-bit block-scaled paged KV cache (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg and its
reference arm) may import this package.  The product library (``block_quantized_bit_gb300``)
never imports it and shares no code with it.
"""
from .oracle import *  # noqa: F401,F403
