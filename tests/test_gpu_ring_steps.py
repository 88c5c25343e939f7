"""Separate-partials mode: one call per ring step writes the step's partial
(O_t, LSE_t); ra_lse_merge combines partials.  Each partial is checked against
the oracle's attention over exactly the keys of shard (r - t) mod N for the
queries of shard r; the merged result against the oracle's full attention, in
ring order and in reverse order."""
import math

import numpy as np
import pytest
import torch

import oracle
from context_ra_forward_gb300 import inputs
from gpu_util import compare, to_orig

pytestmark = pytest.mark.gpu

CASES = [
    # (name, dtype, causal, alibi, N, layout, B, H, S, D)
    ("zz_causal", "bf16", True, False, 4, "zigzag", 1, 2, 2048, 128),
    ("st_alibi", "bf16", True, True, 4, "strided", 1, 2, 4096, 128),
    ("zz_alibi", "bf16", True, True, 4, "zigzag", 1, 2, 4096, 128),   # 512-token chunks
    ("ct_noncausal", "bf16", False, False, 2, "contiguous", 1, 2, 1024, 128),
    ("f32_zz", "f32", True, True, 2, "zigzag", 1, 2, 1024, 64),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_ring_steps_and_merge(case):
    import context_ra_forward_gb300 as ra
    name, dt, causal, alibi, N, layout, B, H, S, D = case
    w = inputs.Workload(name, B, H, S, D, dt, causal, alibi, N, layout, False, 23)
    x = inputs.make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v = (ra.zigzag_permute(x[n].to(dev), N, layout) for n in ("q", "k", "v"))
    sl = inputs.alibi_slopes(H).to(dev) if alibi else None
    f = {n: inputs.to_f64_numpy(t) for n, t in x.items()}
    sl64 = inputs.alibi_slopes(H).double().numpy() if alibi else None
    scale = 1.0 / math.sqrt(D)
    members = oracle.shard_members(S, N, layout)
    c = S // N
    parts = []
    for t in range(N):
        o_t, l_t = ra.forward_ring_step(q, k, v, t, causal=causal, alibi_slopes=sl, N=N, layout=layout)
        parts.append((o_t, l_t))
        for r in range(N):
            rows = np.array(members[r])
            keys = np.array(members[(r - t) % N])
            o_ref, l_ref = oracle.attention_forward(f["q"], f["k"], f["v"], causal=causal, scale=scale,
                                                    slopes=sl64, rows=rows, keys=keys)
            got_o = o_t[:, :, r * c:(r + 1) * c].double().cpu().numpy()
            got_l = l_t[:, :, r * c:(r + 1) * c].double().cpu().numpy()
            compare(got_o, o_ref, dt, f"step {t} shard {r} O")
            compare(got_l, l_ref, dt, f"step {t} shard {r} LSE")
    o_full, l_full = oracle.attention_forward(f["q"], f["k"], f["v"], causal=causal, scale=scale, slopes=sl64)
    perm, _ = oracle.index_maps(S, N, layout)
    for order in (list(range(N)), list(reversed(range(N)))):
        acc_o = parts[order[0]][0].clone()
        acc_l = parts[order[0]][1].clone()
        out = torch.empty((B, H, S, D), dtype=q.dtype, device=dev)
        for j, t in enumerate(order[1:]):
            ra.lse_merge(acc_o, acc_l, parts[t][0], parts[t][1], out=out if j == N - 2 else None)
        if N == 1:
            out.copy_(acc_o.to(q.dtype))
        compare(to_orig(out, perm), o_full, dt, f"merged O, order {order}")
        compare(to_orig(acc_l, perm), l_full, dt, f"merged LSE, order {order}")
    st, detail = ra.check_device_status()
    assert st == 0, detail


def test_ring_step_rejects():
    import context_ra_forward_gb300 as ra
    q = torch.zeros((1, 1, 1200, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ra.RAError) as e:   # 400-slot shards: not a multiple of 256
        ra.forward_ring_step(q, q, q, 0, N=3, layout="contiguous")
    assert e.value.status == -2
    q = torch.zeros((1, 1, 1024, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ra.RAError) as e:
        ra.forward_ring_step(q, q, q, 4, N=4, layout="contiguous")
    assert e.value.status == -1
