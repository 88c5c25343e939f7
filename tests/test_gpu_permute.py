"""ra_zigzag_permute / ra_unpermute on the GPU: bit-exact against the oracle's
index maps (explicit loop construction), for every dtype, head dim and layout."""
import numpy as np
import pytest
import torch

import oracle
from context_ra_forward_gb300 import inputs

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


@pytest.mark.parametrize("dtype,D", [(torch.float32, 64), (torch.float32, 128),
                                     (torch.bfloat16, 64), (torch.bfloat16, 128)])
@pytest.mark.parametrize("S,N,layout", [(1024, 4, "zigzag"), (1200, 3, "zigzag"), (1000, 4, "contiguous"),
                                        (8, 4, "zigzag"), (2, 1, "zigzag"), (4096, 8, "zigzag"),
                                        (768, 1, "contiguous"), (16, 4, "strided"), (1200, 3, "strided"),
                                        (4096, 8, "strided")])
def test_permute_bit_exact(dtype, D, S, N, layout):
    import context_ra_forward_gb300 as ra
    x = inputs.randn((2, 3, S, D), 77 + S, dtype).cuda()
    perm, inv = oracle.index_maps(S, N, layout)
    y = ra.zigzag_permute(x, N, layout)
    want = x[:, :, torch.as_tensor(perm, device=x.device)]
    assert torch.equal(_bits(y), _bits(want))
    z = ra.unpermute(y, N, layout)
    assert torch.equal(_bits(z), _bits(x))
    # unpermute on its own: slot -> original via inv
    w = ra.unpermute(x, N, layout)
    assert torch.equal(_bits(w), _bits(x[:, :, torch.as_tensor(inv, device=x.device)]))


def test_permute_full_size_c5():
    """C5 tensor size (1 x 16 x 262144 x 128 bf16, 1 GiB): exact against the map."""
    import context_ra_forward_gb300 as ra
    w = inputs.WORKLOADS["C5"]
    x = inputs.randn((w.B, w.H, w.S, w.D), 5, torch.bfloat16).cuda()
    perm, _ = oracle.index_maps(w.S, w.N, w.layout)
    y = ra.zigzag_permute(x, w.N, w.layout)
    assert torch.equal(_bits(y), _bits(x[:, :, torch.as_tensor(perm, device=x.device)]))
    assert torch.equal(_bits(ra.unpermute(y, w.N, w.layout)), _bits(x))


def test_permute_empty_is_noop():
    import context_ra_forward_gb300 as ra
    x = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16, device="cuda")
    y = ra.zigzag_permute(x, 4, "zigzag")
    assert y.shape == x.shape
