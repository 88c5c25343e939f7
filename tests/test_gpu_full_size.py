"""Full-size configurations, in the launch configuration the benchmark times.

The oracle cannot evaluate these in full, so each check uses outputs the oracle
computes one by one — forward rows and dQ rows (each needs only its own query
row), dK/dV of the last keys (seen by few queries) — on a head subset that
includes the first and the last head (ALiBi slopes differ per head), plus
properties that hold at any size: sum_j dV_j = sum_i dO_i and sum_j dK_j = 0.
Heads are independent, so a head subset is exact parity on those heads."""
import math

import numpy as np
import pytest
import torch

import oracle
from context_ra_forward_gb300 import inputs
from gpu_util import compare, to_orig

pytestmark = pytest.mark.gpu


def _run(w):
    import context_ra_forward_gb300 as ra
    x = inputs.make_inputs(w)
    dev = torch.device("cuda:0")
    sl = inputs.alibi_slopes(w.H).to(dev) if w.alibi else None
    xp = {n: ra.zigzag_permute(t.to(dev), w.N, w.layout) for n, t in x.items()}
    o, lse = ra.forward(xp["q"], xp["k"], xp["v"], causal=w.causal, alibi_slopes=sl, N=w.N, layout=w.layout)
    res = {"o": ra.unpermute(o, w.N, w.layout), "lse": lse}
    if w.backward:
        g = ra.backward(xp["q"], xp["k"], xp["v"], o, lse, xp["do"], causal=w.causal, alibi_slopes=sl,
                        N=w.N, layout=w.layout)
        res.update({n: ra.unpermute(t, w.N, w.layout) for n, t in zip(("dq", "dk", "dv"), g)})
    st, detail = ra.check_device_status()
    assert st == 0, detail
    return x, res


def _sample_rows(w, count):
    """Query rows from every shard: slots spread over the shard-major buffer."""
    perm, _ = oracle.index_maps(w.S, w.N, w.layout)
    slots = np.linspace(0, w.S - 1, count).astype(np.int64)
    return np.unique(np.concatenate([perm[slots], [0, w.S - 1]]))


@pytest.mark.parametrize("cfg", ["C2", "C3", "C4", "C5", "C3S", "C5S"])
def test_full_size(cfg):
    w = inputs.WORKLOADS[cfg]
    x, res = _run(w)
    scale = 1.0 / math.sqrt(w.D)
    perm, _ = oracle.index_maps(w.S, w.N, w.layout)
    lse_orig = to_orig(res["lse"], perm)
    rows = _sample_rows(w, 48)
    slopes_all = inputs.alibi_slopes(w.H).double().numpy() if w.alibi else None
    for hh in sorted({0, w.H - 1}):
        f = {n: inputs.to_f64_numpy(t[:, hh:hh + 1]) for n, t in x.items()}
        sl = None if slopes_all is None else slopes_all[hh:hh + 1]
        o_ref, l_ref = oracle.attention_forward(f["q"], f["k"], f["v"], causal=w.causal, scale=scale,
                                                slopes=sl, rows=rows)
        o_gpu = res["o"][:, hh:hh + 1, rows].float().cpu().numpy().astype(np.float64)
        compare(o_gpu, o_ref, w.dtype, f"{cfg} head {hh} O rows")
        compare(lse_orig[:, hh:hh + 1, rows], l_ref, w.dtype, f"{cfg} head {hh} LSE rows")
        if not w.backward:
            continue
        dq_ref = oracle.backward_dq_rows(f["q"], f["k"], f["v"], f["do"], rows, causal=w.causal,
                                         scale=scale, slopes=sl)
        dq_gpu = res["dq"][:, hh:hh + 1, rows].float().cpu().numpy().astype(np.float64)
        compare(dq_gpu, dq_ref, w.dtype, f"{cfg} head {hh} dQ rows")
        cols = np.arange(w.S - 192, w.S)
        dk_ref, dv_ref = oracle.backward_dkdv_cols(f["q"], f["k"], f["v"], f["do"], cols, causal=w.causal,
                                                   scale=scale, slopes=sl)
        compare(res["dk"][:, hh:hh + 1, cols].float().cpu().numpy().astype(np.float64), dk_ref, w.dtype,
                f"{cfg} head {hh} dK tail")
        compare(res["dv"][:, hh:hh + 1, cols].float().cpu().numpy().astype(np.float64), dv_ref, w.dtype,
                f"{cfg} head {hh} dV tail")
    if w.backward:
        # properties that hold at any size, on every head
        dv_sum = res["dv"].double().sum(dim=2)
        do_sum = x["do"].to(dv_sum.device).double().sum(dim=2)
        rel = float((dv_sum - do_sum).norm() / do_sum.norm())
        assert rel < 1e-2, f"sum dV vs sum dO: rel {rel:.3e}"
        dk = res["dk"].double()
        ratio = float(dk.sum(dim=2).norm() / dk.abs().sum(dim=2).norm())
        assert ratio < 1e-2, f"sum dK not ~0: ratio {ratio:.3e}"


def test_long_accumulation_dkdv():
    """dK and dV of keys that collect gradient from many query tiles, element by
    element: the 64K-token causal zig-zag layout (N = 8, 16 chunks of 4096) with a
    backward, one head; the 128 keys at global positions S-16384 .. S-16257 are seen
    by 16384 queries each (128 query tiles), spread over both chunks of every
    shard's second half.  Compared with the oracle's dK/dV columns, which recompute
    those 16384 query rows in full."""
    w = inputs.Workload("C3-backward", 1, 1, 65536, 128, "bf16", True, False, 8, "zigzag", True, 3)
    x, res = _run(w)
    scale = 1.0 / math.sqrt(w.D)
    f = {n: inputs.to_f64_numpy(t) for n, t in x.items()}
    cols = np.arange(w.S - 16384, w.S - 16384 + 128)
    dk_ref, dv_ref = oracle.backward_dkdv_cols(f["q"], f["k"], f["v"], f["do"], cols, causal=True, scale=scale)
    compare(res["dk"][:, :, cols].float().cpu().numpy().astype(np.float64), dk_ref, w.dtype, "dK, 16384 queries")
    compare(res["dv"][:, :, cols].float().cpu().numpy().astype(np.float64), dv_ref, w.dtype, "dV, 16384 queries")
