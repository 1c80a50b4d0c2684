"""GB300-native SMOE group-quantised routed-expert MoE layer.

The compute path lives in the C-ABI library ``libsmoe.so`` (hand-written CUDA
for sm_103a, declared in ``include/smoe.h``); ``bit_expert_weight_gb300.smoe``
is its thin ctypes binding.  Importing this package loads nothing: the
binding loads the library on first use and raises if it is missing.
"""

__all__ = ["smoe", "synth"]
