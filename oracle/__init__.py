"""fp64 CPU oracle for exact attention, forward and backward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs use this package.  It shares no code with the CUDA library.
"""
from .attention import (  # noqa: F401
    attention,
    attention_rows,
    attention_weights,
    merge_max_sum,
    merge_partials,
    online_max_sum,
    softmax_safe,
    tiled_attention,
)
from . import fp8  # noqa: F401
from .attention_backward import (  # noqa: F401
    attention_backward,
    rowdot,
    tiled_attention_backward,
)
