"""Run-to-run comparison as a race check: the same inputs, launched again, must give
the same results.  The forward, dK and dV have no cross-CTA accumulation (each
CTA owns its query pair or its K/V tile and works in a fixed order), so they are
compared bit for bit; dQ is summed in fp32 by reduce-adds whose order between
CTAs is not fixed, so it may differ by the rounding of that order only.  A race
on shared or tensor memory (a buffer refilled before it was read, a barrier
phase taken too early) shows up as a larger difference."""
import pytest
import torch

from context_ra_forward_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = [
    # (S, H, N, layout, causal, alibi)
    (16384, 4, 8, "zigzag", True, False),
    (16384, 4, 8, "strided", True, False),
    (8192, 4, 4, "contiguous", True, True),
    (8192, 2, 2, "zigzag", False, False),
    (1200, 2, 3, "zigzag", True, True),     # ragged runs: 200-token chunks on the tensor cores
]


@pytest.mark.parametrize("S,H,N,layout,causal,alibi", CASES,
                         ids=[f"{c[3]}_S{c[0]}_{'causal' if c[4] else 'full'}{'_alibi' if c[5] else ''}" for c in CASES])
def test_repeated_runs_agree(S, H, N, layout, causal, alibi):
    import context_ra_forward_gb300 as ra
    w = inputs.Workload("det", 1, H, S, 128, "bf16", causal, alibi, N, layout, True, 77)
    x = inputs.make_inputs(w)
    d = torch.device("cuda:0")
    q, k, v, do = (ra.zigzag_permute(x[n].to(d), N, layout) for n in ("q", "k", "v", "do"))
    sl = inputs.alibi_slopes(H).to(d) if alibi else None
    runs = []
    for _ in range(3):
        o, lse = ra.forward(q, k, v, causal=causal, alibi_slopes=sl, N=N, layout=layout)
        dq, dk, dv = ra.backward(q, k, v, o, lse, do, causal=causal, alibi_slopes=sl, N=N, layout=layout)
        runs.append((o, lse, dq, dk, dv))
    st, detail = ra.check_device_status()
    assert st == 0, detail
    o0, lse0, dq0, dk0, dv0 = runs[0]
    for o, lse, dq, dk, dv in runs[1:]:
        assert torch.equal(o.view(torch.int16), o0.view(torch.int16)), "O differs between runs"
        assert torch.equal(lse.view(torch.int32), lse0.view(torch.int32)), "LSE differs between runs"
        assert torch.equal(dk.view(torch.int16), dk0.view(torch.int16)), "dK differs between runs"
        assert torch.equal(dv.view(torch.int16), dv0.view(torch.int16)), "dV differs between runs"
        # dQ: fp32 sums in another order, then one bf16 rounding: a few bf16 ulps at most
        a, b = dq.float(), dq0.float()
        bound = 2.0 ** -6 * torch.maximum(a.abs(), b.abs()) + 1e-6
        worst = float(((a - b).abs() - bound).max())
        assert worst <= 0.0, f"dQ differs between runs beyond reduction-order rounding ({worst:.3e})"
