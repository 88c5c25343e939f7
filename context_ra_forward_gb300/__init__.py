"""Ring / zig-zag blockwise exact attention on one GB300 (sm_103a).

The computation lives in the CUDA library libra.so (C ABI: include/ra.h); this
package is its thin Python binding plus the build step and the seeded synthetic
input generators.  The library is loaded on first use; every call raises if it
is missing.
"""
from .binding import (  # noqa: F401
    RAError, LAYOUTS, index_map, zigzag_permute, unpermute, forward, backward,
    backward_workspace_bytes, forward_path, check_device_status, debug_wait_timeout, lib,
    kernel_launch_count, backward_noalloc, noalloc_scratch_bytes, debug_wait_sites,
    forward_ring_step, lse_merge, forward_fp8, rope_permute, rope_unpermute, shard_work,
    backward_path,
)
