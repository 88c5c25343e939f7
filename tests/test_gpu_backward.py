"""ra_backward on the GPU against the oracle's analytic gradient."""
import numpy as np
import pytest

import oracle
from context_ra_forward_gb300 import inputs
from gpu_util import compare, run_case

pytestmark = pytest.mark.gpu

CASES = [
    # (name, dtype, causal, alibi, N, layout, B, H, S, D)
    ("c5_reduced", "bf16", True, False, 16, "zigzag", 1, 2, 4096, 128),
    ("c5_alibi", "bf16", True, True, 4, "zigzag", 1, 2, 2048, 128),
    ("noncausal", "bf16", False, False, 2, "contiguous", 1, 2, 1024, 128),
    ("ragged", "bf16", True, False, 3, "zigzag", 1, 2, 1200, 128),
    ("tail", "bf16", True, True, 4, "contiguous", 1, 1, 1000, 128),
    ("d64", "bf16", True, False, 2, "zigzag", 1, 2, 512, 64),
    ("f32", "f32", True, True, 4, "zigzag", 1, 2, 1024, 64),
    ("strided", "bf16", True, False, 8, "strided", 1, 2, 2048, 128),
    ("strided_alibi", "bf16", True, True, 4, "strided", 1, 2, 2048, 128),
    ("strided_nc_alibi", "bf16", False, True, 2, "strided", 1, 1, 1024, 128),
    ("strided_ragged", "bf16", True, False, 3, "strided", 1, 2, 1200, 128),
    ("strided_odd", "bf16", True, True, 4, "strided", 1, 2, 1292, 128),   # S % N == 0, S % 2N != 0
    # several batches and heads (per-(b, h) block order, per-head ALiBi slopes)
    ("batch_heads", "bf16", True, True, 2, "zigzag", 2, 3, 1024, 128),
    ("batch_heads_nc", "bf16", False, False, 4, "contiguous", 3, 2, 512, 128),
    # fp32 (CUDA-core path) with a ragged tail and a strided layout
    ("f32_ragged", "f32", True, False, 3, "zigzag", 1, 2, 600, 64),
    ("f32_strided", "f32", True, True, 4, "strided", 2, 1, 512, 128),
    # ragged runs on the tensor cores: tiles meeting a run boundary, a partial last
    # tile, rows whose 16-byte alignment depends on the head (S % 4 != 0)
    ("ragged_alibi", "bf16", True, True, 3, "zigzag", 1, 2, 1200, 128),
    ("ragged_nc", "bf16", False, False, 3, "zigzag", 2, 1, 1200, 128),
    ("odd_rows", "bf16", True, True, 2, "contiguous", 1, 3, 1002, 128),
    ("short_runs", "bf16", True, False, 4, "zigzag", 1, 2, 512, 128),  # 64-token chunks: CUDA cores
]

# the kernel each bf16 case runs: ragged runs of >= 128 slots take the tensor cores
PATHS = {"ragged": 1, "tail": 1, "strided_ragged": 1, "strided_odd": 1, "ragged_alibi": 1, "ragged_nc": 1,
         "odd_rows": 1, "c5_reduced": 1, "short_runs": 2, "f32": 2}


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_parity(case):
    import torch
    import context_ra_forward_gb300 as ra
    name, dt, causal, alibi, N, layout, B, H, S, D = case
    if name in PATHS:
        tdt = torch.bfloat16 if dt == "bf16" else torch.float32
        assert ra.backward_path(B, H, S, D, tdt, N, layout) == PATHS[name], name
    w = inputs.Workload(name, B, H, S, D, dt, causal, alibi, N, layout, True, 17)
    out, f64, slopes, scale = run_case(w)
    dq, dk, dv = oracle.attention_backward(f64["q"], f64["k"], f64["v"], f64["do"], causal=causal,
                                           scale=scale, slopes=slopes)
    compare(out["dq"], dq, dt, "dQ")
    compare(out["dk"], dk, dt, "dK")
    compare(out["dv"], dv, dt, "dV")


def test_backward_empty_problem():
    """S = 0: nothing to compute, nothing launched, empty gradients returned."""
    import torch
    import context_ra_forward_gb300 as ra
    q = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 2, 0), dtype=torch.float32, device="cuda")
    before = ra.kernel_launch_count()
    dq, dk, dv = ra.backward(q, q, q, q, lse, q, causal=True, N=4, layout="zigzag")
    assert ra.kernel_launch_count() == before
    assert dq.shape == dk.shape == dv.shape == q.shape
