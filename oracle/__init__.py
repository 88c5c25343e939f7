"""fp64 CPU oracle for ring / zig-zag blockwise attention — TEST INFRASTRUCTURE ONLY.

Only tests/, the package's smoke check (__graft_entry__.smoke) and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library and the library never calls it.
"""
from .attention import (  # noqa: F401
    CONTIGUOUS, ZIGZAG, STRIDED, LAYOUTS, check_split, shard_members, index_maps,
    causal_pairs_per_shard, attention_forward, attention_backward,
    backward_dq_rows, backward_dkdv_cols, lse_merge, ring_forward,
    online_softmax_rows,
)
from .rope import rope_frequencies, rope_rotate  # noqa: F401
