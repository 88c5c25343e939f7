"""ra_forward on the GPU against the fp64 oracle, element by element, on seeded
inputs; cross-layout and cross-N consistency; edge cases."""
import math

import numpy as np
import pytest
import torch

import oracle
from context_ra_forward_gb300 import inputs
from gpu_util import compare, run_case, to_orig

pytestmark = pytest.mark.gpu

W = inputs.WORKLOADS


def _check_forward(w, **sizes):
    out, f64, slopes, scale = run_case(w, backward=False, **sizes)
    o_ref, l_ref = oracle.attention_forward(f64["q"], f64["k"], f64["v"], causal=w.causal,
                                            scale=scale, slopes=slopes)
    a = compare(out["o"], o_ref, w.dtype, "O")
    b = compare(out["lse"], l_ref, w.dtype, "LSE")
    return a, b


def test_c1_full_fp32():
    """C1 in full: fp32, causal, B1 H2 S1024 D64, N=4 zig-zag; max abs <= 1e-4."""
    _check_forward(W["C1"])


@pytest.mark.parametrize("cfg,S,H", [("C2", 2048, 2), ("C3", 2048, 2), ("C4", 2048, 3), ("C4", 4096, 4),
                                     ("C5", 4096, 1)])
def test_bf16_reduced(cfg, S, H):
    """The bf16 configurations at a size the oracle finishes in seconds (same
    layout and N, several tiles per shard).  C4 at S=2048 has 128-token chunks
    (the per-element ALiBi path); at S=4096 its 256-token chunks take the path
    that adds the ALiBi column term on the tensor core."""
    _check_forward(W[cfg], S=S, H=H)


@pytest.mark.parametrize("layout,N,S,slopes", [
    ("zigzag", 4, 2048, [0.9, 40.0, 2.0 ** -8]),   # head 1: too steep for the tensor-core term
    ("strided", 8, 4096, [0.9, 3.0]),               # step 8: head 1 too steep
    ("contiguous", 2, 1024, [1.0, -0.25]),          # a negative slope (a bias growing with distance)
])
def test_alibi_caller_slopes(layout, N, S, slopes):
    """Causal ALiBi with slopes the caller chooses, including ones steep enough
    that the kernel keeps the per-element bias for that head while the other
    heads of the same launch add the column term on the tensor core."""
    import context_ra_forward_gb300 as ra
    H = len(slopes)
    w = inputs.Workload("sl", 1, H, S, 128, "bf16", True, True, N, layout, False, 29)
    x = inputs.make_inputs(w)
    d = torch.device("cuda:0")
    q, k, v = (ra.zigzag_permute(x[n].to(d), N, layout) for n in ("q", "k", "v"))
    sl = torch.tensor(slopes, dtype=torch.float32)
    o, lse = ra.forward(q, k, v, causal=True, alibi_slopes=sl.to(d), N=N, layout=layout)
    perm, _ = oracle.index_maps(S, N, layout)
    f = {n: inputs.to_f64_numpy(t) for n, t in x.items()}
    o_ref, l_ref = oracle.attention_forward(f["q"], f["k"], f["v"], causal=True, scale=1.0 / math.sqrt(128),
                                            slopes=sl.double().numpy())
    compare(to_orig(o, perm), o_ref, "bf16", "O")
    compare(to_orig(lse, perm), l_ref, "bf16", "LSE")


RAGGED = [
    # (name, dtype, causal, alibi, N, layout, B, H, S, D)
    ("zz_h200", "bf16", True, False, 3, "zigzag", 1, 2, 1200, 128),     # chunks of 200: tiles straddle
    ("ct_c250", "bf16", True, True, 4, "contiguous", 2, 1, 1000, 128),  # ragged tail (1000 % 128)
    ("zz_h1", "bf16", True, True, 4, "zigzag", 1, 2, 8, 128),           # one token per chunk
    ("tiny", "bf16", False, False, 1, "zigzag", 1, 1, 2, 128),
    ("nc_alibi", "bf16", False, True, 2, "zigzag", 1, 2, 640, 128),     # symmetric ALiBi
    ("d64_bf16", "bf16", True, True, 2, "zigzag", 1, 2, 512, 64),
    ("f32_d128", "f32", True, True, 2, "zigzag", 1, 2, 384, 128),
    ("f32_nc", "f32", False, False, 3, "contiguous", 1, 2, 300, 64),
    ("n_eq_half_s", "bf16", True, False, 64, "zigzag", 1, 1, 256, 128),  # chunk = 2 tokens
    ("batch_heads", "bf16", True, False, 2, "zigzag", 3, 5, 512, 128),
    # tiles whose visible keys are a column prefix (no ALiBi): ragged tails, diagonals
    ("nc_ragged", "bf16", False, False, 2, "contiguous", 1, 2, 1000, 128),  # last key tile 104 wide
    ("ct_ragged_causal", "bf16", True, False, 4, "contiguous", 1, 2, 1000, 128),
    ("st_ragged_causal", "bf16", True, False, 3, "strided", 1, 2, 1200, 128),
    # token-strided layout: shard r holds tokens r, r+N, ...
    ("st_aligned", "bf16", True, False, 4, "strided", 1, 2, 2048, 128),     # 512 slots per shard
    ("st_alibi", "bf16", True, True, 8, "strided", 1, 2, 4096, 128),
    ("st_nc_alibi", "bf16", False, True, 2, "strided", 1, 2, 1024, 128),
    ("st_ragged", "bf16", True, True, 3, "strided", 1, 2, 1200, 128),      # 400 slots: tiles straddle shards
    ("st_odd", "bf16", True, True, 4, "strided", 1, 2, 1292, 128),         # S % N == 0, S % 2N != 0
    ("st_odd_nc", "bf16", False, False, 4, "strided", 1, 2, 1292, 128),
    ("st_f32", "f32", True, True, 4, "strided", 1, 2, 512, 64),
]


@pytest.mark.parametrize("case", RAGGED, ids=[c[0] for c in RAGGED])
def test_edge_cases(case):
    name, dt, causal, alibi, N, layout, B, H, S, D = case
    w = inputs.Workload(name, B, H, S, D, dt, causal, alibi, N, layout, False, 13)
    _check_forward(w)


def test_layout_and_n_independence():
    """O and LSE in original order do not depend on N or the layout (the ring is
    a visit order; the merge is exact up to rounding)."""
    base = None
    for N, layout in [(1, "contiguous"), (8, "zigzag"), (4, "contiguous"), (16, "zigzag"), (8, "strided")]:
        w = inputs.Workload("x", 1, 2, 4096, 128, "bf16", True, False, N, layout, False, 21)
        out, _, _, _ = run_case(w, backward=False)
        if base is None:
            base = out
            continue
        for n in ("o", "lse"):
            assert np.max(np.abs(out[n] - base[n])) <= 2e-2


def test_custom_scale():
    w = inputs.Workload("s", 1, 2, 512, 128, "bf16", True, False, 2, "zigzag", False, 3)
    import context_ra_forward_gb300 as ra
    x = inputs.make_inputs(w)
    q, k, v = (ra.zigzag_permute(x[n].cuda(), w.N, w.layout) for n in ("q", "k", "v"))
    o, lse = ra.forward(q, k, v, causal=True, softmax_scale=0.05, N=w.N, layout=w.layout)
    perm, _ = oracle.index_maps(w.S, w.N, w.layout)
    f = {n: inputs.to_f64_numpy(t) for n, t in x.items()}
    o_ref, l_ref = oracle.attention_forward(f["q"], f["k"], f["v"], causal=True, scale=0.05)
    compare(to_orig(o, perm), o_ref, "bf16", "O")
    compare(to_orig(lse, perm), l_ref, "bf16", "LSE")


def test_empty_problem():
    import context_ra_forward_gb300 as ra
    q = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16, device="cuda")
    o, lse = ra.forward(q, q, q, causal=True, N=4, layout="zigzag")
    assert o.shape == q.shape and lse.shape == (1, 2, 0)


def test_rejects_bad_arguments():
    import context_ra_forward_gb300 as ra
    q = torch.zeros((1, 2, 1000, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ra.RAError) as e:
        ra.forward(q, q, q, causal=True, N=3, layout="zigzag")  # 1000 % 6
    assert e.value.status == -1
    q96 = torch.zeros((1, 2, 64, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ra.RAError) as e:
        ra.forward(q96, q96, q96, N=1)
    assert e.value.status == -2


def test_non_finite_input_propagates():
    """A NaN in K reaches every row that sees it and no other (exact masking)."""
    import context_ra_forward_gb300 as ra
    w = inputs.Workload("nan", 1, 1, 512, 128, "bf16", True, False, 2, "contiguous", False, 4)
    x = inputs.make_inputs(w)
    x["k"][0, 0, 300, 5] = float("nan")
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))  # N=2 contiguous: identity map
    o, lse = ra.forward(q, k, v, causal=True, N=2, layout="contiguous")
    bad = torch.isnan(o[0, 0]).any(dim=-1).cpu().numpy()
    assert not bad[:300].any() and bad[300:].all()
