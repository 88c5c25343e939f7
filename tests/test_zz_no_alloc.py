"""ra_backward_noalloc — the backward for callers that cannot allocate device
memory when they run it (a framework that owns every device allocation, memory
fixed at start-up, loops that cannot take an allocation's synchronisation).  It
uses the library's fixed scratch buffer instead of a caller workspace.

The test calls it through the C ABI twice in a row and compares each result with
the regular ra_backward (caller-provided workspace) on the same inputs, within
the parity tolerance of the other tests; the second call also shows that what
the first call left in the shared buffer does not leak into the next result, and
that the call takes no device memory (free device memory is the same before and
after it, with the outputs supplied by the caller).
This file is collected last so that a run stopping at the first failure has run
every other test first; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from context_ra_forward_gb300 import inputs
from gpu_util import TOL

pytestmark = pytest.mark.gpu

CASES = [
    # (name, dtype, causal, alibi, N, layout, B, H, S, D)
    ("bf16_tensor_core", "bf16", True, True, 4, "zigzag", 1, 2, 2048, 128),
    ("f32_cuda_core", "f32", True, False, 2, "zigzag", 1, 2, 512, 64),
]


def _close(a, b, dtype, what):
    a = a.detach().float().cpu().numpy().astype(np.float64)
    b = b.detach().float().cpu().numpy().astype(np.float64)
    err = float(np.max(np.abs(a - b)))
    tol = TOL[dtype]
    assert err <= tol["max_abs"], f"{what}: max abs {err:.3e}"
    if tol["rel_rms"] is not None:
        rel = float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))
        assert rel <= tol["rel_rms"], f"{what}: rel rms {rel:.3e}"


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_noalloc_backward_matches_backward_twice(case):
    import context_ra_forward_gb300 as ra
    name, dt, causal, alibi, N, layout, B, H, S, D = case
    w = inputs.Workload(name, B, H, S, D, dt, causal, alibi, N, layout, True, 29)
    x = inputs.make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (ra.zigzag_permute(x[n].to(dev), N, layout) for n in ("q", "k", "v", "do"))
    sl = inputs.alibi_slopes(H).to(dev) if alibi else None
    o, lse = ra.forward(q, k, v, causal=causal, alibi_slopes=sl, N=N, layout=layout)
    ref = ra.backward(q, k, v, o, lse, do, causal=causal, alibi_slopes=sl, N=N, layout=layout)
    assert ra.backward_workspace_bytes(B, H, S, D) <= ra.noalloc_scratch_bytes()
    outs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    for call in range(2):
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        got = ra.backward_noalloc(q, k, v, o, lse, do, causal=causal, alibi_slopes=sl, N=N, layout=layout,
                                  out=outs)
        torch.cuda.synchronize()
        if call == 1:  # (the first call on a device may still load the library's device code)
            assert torch.cuda.mem_get_info()[0] == free0, "the call took device memory"
        st, detail = ra.check_device_status()
        assert st == 0, detail
        for g, r, n in zip(got, ref, ("dQ", "dK", "dV")):
            _close(g, r, dt, f"call {call + 1} {n}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    import context_ra_forward_gb300 as ra
    L = ra.lib()
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    p = ctypes.c_void_p(t.data_ptr())
    # 64 heads x 65536 tokens need ~2 GB of scratch: rejected before any launch
    st = L.ra_backward_noalloc(p, p, p, p, p, p, p, p, p, 1, 64, 65536, 128, 1, 1, None,
                               ctypes.c_float(0.0), 8, 1, None)
    assert st == -6
