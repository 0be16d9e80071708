"""Float64 CPU oracle for exact tiled attention (test infrastructure only).

Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline leg of bench.py
may import this package; the CUDA library never does.  See attention.py for
the definitions, their sources and their pins.
"""
from .attention import (  # noqa: F401
    attention_flops,
    causal_tile_pairs,
    flash_backward_tiled,
    flash_forward_tiled,
    key_rows_bwd,
    online_softmax,
    rows_fwd_bwd,
    standard_attention_bwd,
    standard_attention_fwd,
    visible_pairs,
)
