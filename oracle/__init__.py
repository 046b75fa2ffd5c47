"""fp64 CPU oracle for blockwise exact attention and the blockwise
feed-forward layer (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA product path never imports,
links or calls it; the two share no code.
"""
from .attention import (  # noqa: F401
    attention_fwd,
    attention_probs,
    attention_bwd,
    attention_rows,
    attention_bwd_by_row_blocks,
    attention_varlen,
    varlen_rows,
    block_state,
    merge_states,
    finalize_state,
    ring_fwd_blocked,
    ring_fwd_blocked_striped,
    striped_positions,
    ring_schedule,
)
from .ffn import (  # noqa: F401
    gelu,
    gelu_grad,
    ffn_fwd,
    ffn_bwd,
    ffn_blocked,
    ffn_bwd_blocked,
)
