"""CPU oracle for the SMOE routed-expert MoE layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or executes anything in here.
"""
from .oracle import *  # noqa: F401,F403
