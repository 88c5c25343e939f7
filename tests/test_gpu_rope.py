"""ra_rope_permute / ra_rope_unpermute on the GPU against the fp64 RoPE oracle
([LC] "超长上下文技术" §2.1.3), element by element, for every dtype, head dim and
layout; the composition with ring attention forward and backward; full C5 size on
sampled rows.

Tolerances (the rotation is a single rounding step, no accumulation): fp32 max abs
1e-5 (cos/sin carry a few 1e-7, times |x| <= ~6); bf16 |delta| <= 2^-8 |ref| + 1e-5
(half a bf16 ulp of the rounded result, plus the fp32 rotation error)."""
import math

import numpy as np
import pytest
import torch

import oracle
from context_ra_forward_gb300 import inputs
from gpu_util import compare, to_orig

pytestmark = pytest.mark.gpu


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _check(got, ref, dt, what):
    err = np.abs(got - ref)
    if dt == torch.float32:
        assert float(err.max()) <= 1e-5, f"{what}: max abs {err.max():.3e}"
    else:
        bound = 2.0 ** -8 * np.abs(ref) + 1e-5
        worst = float(np.max(err - bound))
        assert worst <= 0.0, f"{what}: exceeds the one-rounding bound by {worst:.3e}"


CASES = [
    # (S, N, layout, pos0)
    (1024, 4, "zigzag", 0),
    (1200, 3, "zigzag", 0),          # chunks of 200 tokens
    (1000, 4, "contiguous", 77),
    (1200, 3, "strided", 0),
    (4096, 8, "strided", 5000),
    (8, 4, "zigzag", 0),             # one token per chunk
    (2, 1, "contiguous", 0),
    (2048, 16, "zigzag", 2 ** 31 - 2048),  # the largest positions allowed
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S,N,layout,pos0", CASES, ids=[f"{c[2]}_S{c[0]}_N{c[1]}_p{c[3]}" for c in CASES])
def test_rope_permute_parity(dtype, D, S, N, layout, pos0):
    import context_ra_forward_gb300 as ra
    x = inputs.randn((2, 3, S, D), 300 + S + D, dtype).cuda()
    perm, inv = oracle.index_maps(S, N, layout)
    pos = np.arange(S, dtype=np.float64) + pos0
    ref = oracle.rope_rotate(_f64(x), pos)[:, :, perm]        # rotated, then shard-major
    y = ra.rope_permute(x, N, layout, pos0=pos0)
    _check(_f64(y), ref, dtype, "rope_permute")
    # the transpose, on its own input (a shard-major tensor)
    z = ra.rope_unpermute(x, N, layout, pos0=pos0)
    ref_t = oracle.rope_rotate(_f64(x)[:, :, inv], pos, inverse=True)
    _check(_f64(z), ref_t, dtype, "rope_unpermute")
    # round trip: the inverse of the prologue
    if dtype == torch.float32:
        back = ra.rope_unpermute(y, N, layout, pos0=pos0)
        assert float((back - x).abs().max()) <= 1e-5


def test_rope_base_and_bf16_positions():
    """Another base (500000), and position 0 is the identity, bit for bit."""
    import context_ra_forward_gb300 as ra
    S, N = 2048, 4
    x = inputs.randn((1, 2, S, 128), 9, torch.bfloat16).cuda()
    perm, _ = oracle.index_maps(S, N, "zigzag")
    y = ra.rope_permute(x, N, "zigzag", base=500000.0, pos0=123)
    ref = oracle.rope_rotate(_f64(x), np.arange(S) + 123.0, base=500000.0)[:, :, perm]
    _check(_f64(y), ref, torch.bfloat16, "base 500000")
    y0 = ra.rope_permute(x, 1, "contiguous")
    assert torch.equal(y0[:, :, 0].view(torch.int16), x[:, :, 0].view(torch.int16))


@pytest.mark.parametrize("layout,N", [("zigzag", 4), ("strided", 4)])
def test_rope_with_attention(layout, N):
    """The fused prologue composed with ring attention, forward and backward:
    O = attention(R q, R k, v); the gradients of the caller's q and k are
    R^T dQ_rot and R^T dK_rot (ra_rope_unpermute)."""
    import context_ra_forward_gb300 as ra
    w = inputs.Workload("rope", 1, 2, 2048, 128, "bf16", True, False, N, layout, True, 61)
    x = inputs.make_inputs(w)
    d = torch.device("cuda:0")
    q = ra.rope_permute(x["q"].to(d), N, layout)
    k = ra.rope_permute(x["k"].to(d), N, layout)
    v = ra.zigzag_permute(x["v"].to(d), N, layout)
    do = ra.zigzag_permute(x["do"].to(d), N, layout)
    o, lse = ra.forward(q, k, v, causal=True, N=N, layout=layout)
    dq, dk, dv = ra.backward(q, k, v, o, lse, do, causal=True, N=N, layout=layout)
    dq_o = ra.rope_unpermute(dq, N, layout)
    dk_o = ra.rope_unpermute(dk, N, layout)
    st, detail = ra.check_device_status()
    assert st == 0, detail

    f = {n: inputs.to_f64_numpy(t) for n, t in x.items()}
    pos = np.arange(w.S, dtype=np.float64)
    qr, kr = oracle.rope_rotate(f["q"], pos), oracle.rope_rotate(f["k"], pos)
    scale = 1.0 / math.sqrt(w.D)
    o_ref, l_ref = oracle.attention_forward(qr, kr, f["v"], causal=True, scale=scale)
    dqr, dkr, dv_ref = oracle.attention_backward(qr, kr, f["v"], f["do"], causal=True, scale=scale)
    dq_ref = oracle.rope_rotate(dqr, pos, inverse=True)
    dk_ref = oracle.rope_rotate(dkr, pos, inverse=True)
    perm, _ = oracle.index_maps(w.S, N, layout)
    compare(to_orig(o, perm), o_ref, "bf16", "O")
    compare(to_orig(lse, perm), l_ref, "bf16", "LSE")
    compare(to_orig(dv, perm), dv_ref, "bf16", "dV")
    compare(_f64(dq_o), dq_ref, "bf16", "dQ (caller's q)")
    compare(_f64(dk_o), dk_ref, "bf16", "dK (caller's k)")


def test_rope_full_size_c5():
    """C5 tensor size (1 x 16 x 262144 x 128 bf16): rows from every shard and both
    ends, on every head, against the oracle; the transpose restores x."""
    import context_ra_forward_gb300 as ra
    w = inputs.WORKLOADS["C5"]
    x = inputs.randn((w.B, w.H, w.S, w.D), 8, torch.bfloat16).cuda()
    y = ra.rope_permute(x, w.N, w.layout)
    perm, _ = oracle.index_maps(w.S, w.N, w.layout)
    slots = np.unique(np.concatenate([np.linspace(0, w.S - 1, 96).astype(np.int64), [0, w.S - 1]]))
    g = perm[slots]
    xs = _f64(x[:, :, torch.as_tensor(g, device=x.device)])
    ref = oracle.rope_rotate(xs, g.astype(np.float64))
    _check(_f64(y[:, :, torch.as_tensor(slots, device=x.device)]), ref, torch.bfloat16, "C5 rows")
    back = ra.rope_unpermute(y, w.N, w.layout)
    # two bf16 roundings.  The first one's error vector in a pair (i, i + D/2) has
    # length <= 2^-8 r (r = the pair's length, kept by the rotation) and is rotated
    # back into both features; the second adds half an ulp of the result:
    # |back_i - x_i| <= 2^-8 (r + |x_i|) (1 + 2^-8) + 1e-5.
    xf = x.float()
    r = torch.sqrt(xf[..., :64] ** 2 + xf[..., 64:] ** 2).repeat(1, 1, 1, 2)
    bound = 2.0 ** -8 * (r + xf.abs()) * (1 + 2.0 ** -8) + 1e-5
    assert bool(((back.float() - xf).abs() <= bound).all())


def test_rope_rejects_bad_arguments():
    import context_ra_forward_gb300 as ra
    x = torch.zeros((1, 2, 1024, 128), dtype=torch.bfloat16, device="cuda")
    for kw, status in (({"base": 1.0}, -1), ({"base": float("nan")}, -1), ({"pos0": -1}, -1),
                       ({"pos0": 2 ** 31 - 1000}, -1)):
        with pytest.raises(ra.RAError) as e:
            ra.rope_permute(x, 4, "zigzag", **kw)
        assert e.value.status == status, kw
    with pytest.raises(ra.RAError) as e:
        ra.rope_permute(x, 4, "zigzag", out=x)        # in place: overlapping buffers
    assert e.value.status == -1
    x8 = torch.zeros((1, 2, 1024, 128), dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(ra.RAError) as e:
        ra.rope_permute(x8, 4, "zigzag")
    assert e.value.status == -2
    empty = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16, device="cuda")
    assert ra.rope_permute(empty, 4, "zigzag").shape == empty.shape
