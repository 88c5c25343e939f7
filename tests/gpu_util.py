"""Helpers for the GPU parity tests: run the library through its binding on
seeded inputs and bring results back to original order via the oracle's map."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from context_ra_forward_gb300 import inputs

# Tolerances fixed for this method's parity: fp32 max abs 1e-4; bf16 max abs 2e-2
# and relative RMS 5e-3 (on O, LSE, dQ, dK, dV).
TOL = {"f32": dict(max_abs=1e-4, rel_rms=None), "bf16": dict(max_abs=2e-2, rel_rms=5e-3)}


def dev():
    return torch.device("cuda:0")


def to_orig(t: torch.Tensor, perm: np.ndarray, axis: int = 2) -> np.ndarray:
    """Shard-major -> original order: slot p holds global position perm[p]."""
    a = t.detach().float().cpu().numpy().astype(np.float64)
    out = np.empty_like(a)
    idx = [slice(None)] * a.ndim
    idx[axis] = perm
    out[tuple(idx)] = a
    return out


def compare(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "") -> dict:
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: non-finite pattern differs"
    # where the reference is not finite (the -inf LSE of a row that sees no key)
    # the result must be the same infinity
    assert np.array_equal(got[~fin], ref[~fin]), f"{what}: non-finite values differ"
    err = np.zeros_like(ref)
    np.subtract(got, ref, out=err, where=fin)
    max_abs = float(np.max(np.abs(err))) if err.size else 0.0
    nref = float(np.linalg.norm(np.where(fin, ref, 0.0)))
    rel = float(np.linalg.norm(err) / nref) if nref > 0 else 0.0
    tol = TOL[dtype]
    assert max_abs <= tol["max_abs"], f"{what}: max abs {max_abs:.3e} > {tol['max_abs']}"
    if tol["rel_rms"] is not None:
        assert rel <= tol["rel_rms"], f"{what}: rel rms {rel:.3e} > {tol['rel_rms']}"
    return {"max_abs": max_abs, "rel_rms": rel}


def run_case(w: inputs.Workload, *, B=None, H=None, S=None, D=None, backward=None):
    """Run permute -> forward (-> backward) on the GPU for a (possibly shrunk)
    workload; returns the GPU results in ORIGINAL order plus the f64 inputs."""
    import context_ra_forward_gb300 as ra
    B = w.B if B is None else B
    H = w.H if H is None else H
    S = w.S if S is None else S
    D = w.D if D is None else D
    bwd = w.backward if backward is None else backward
    wl = inputs.Workload(w.name, B, H, S, D, w.dtype, w.causal, w.alibi, w.N, w.layout, bwd, w.seed)
    x = inputs.make_inputs(wl)
    slopes = inputs.alibi_slopes(H) if w.alibi else None
    d = dev()
    q, k, v = (ra.zigzag_permute(x[n].to(d), w.N, w.layout) for n in ("q", "k", "v"))
    sl_d = slopes.to(d) if slopes is not None else None
    o, lse = ra.forward(q, k, v, causal=w.causal, alibi_slopes=sl_d, N=w.N, layout=w.layout)
    res = {"o": o, "lse": lse}
    if bwd:
        do = ra.zigzag_permute(x["do"].to(d), w.N, w.layout)
        dq, dk, dv = ra.backward(q, k, v, o, lse, do, causal=w.causal, alibi_slopes=sl_d,
                                 N=w.N, layout=w.layout)
        res.update(dq=dq, dk=dk, dv=dv)
    st, detail = ra.check_device_status()
    assert st == 0, f"device status {st} {detail}"
    perm, _ = oracle.index_maps(S, w.N, w.layout)
    out = {n: to_orig(t, perm) for n, t in res.items()}
    f64 = {n: inputs.to_f64_numpy(t) for n, t in x.items()}
    return out, f64, (None if slopes is None else slopes.double().numpy()), 1.0 / math.sqrt(D)
