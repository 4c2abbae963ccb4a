"""GB300-native fused exact attention forward (bf16 in/out, fp32 logsumexp).

The compute path is the C-ABI library ``libfa_gb300.so`` built from ``csrc/``
(hand-written CUDA for sm_103a).  ``fa`` is its thin ctypes binding; importing
it does not need a GPU, but every compute call does, and there is no CPU
fallback: a missing library raises.
"""
__version__ = "0.1.0"
