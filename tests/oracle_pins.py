"""Pins for the fp64 oracle: checks against what the pages and the mathematics fix,
independent of the oracle's own code.

Each pin takes the oracle module as an argument so that the planted-mistake test
(test_oracle_mutations.py) can run the same pins against deliberately broken
copies of the oracle and require that every planted mistake is caught.

Pages cited:
  [CP]  "百万Token上下文训练的挑战与突破" §2.1 (contiguous split), §3.1 (ring)
  [ZZ]  "大模型如何訓練百萬 Token 上下文：上下文并行與 Ring Attention" §Zig Zag Ring Attention
  [LC]  "超长上下文技术" survey §2.1.2 (ALiBi), §2.1.3 (RoPE), §3.1.2 (online softmax)
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _qkv(B, H, S, D, seed):
    r = _rng(seed)
    return (r.standard_normal((B, H, S, D)), r.standard_normal((B, H, S, D)),
            r.standard_normal((B, H, S, D)))


def _slopes(H):
    # the fixture-checked formula of [LC] §2.1.2, restated here for the pins
    return np.array([2.0 ** (-8.0 * i / H) for i in range(1, H + 1)])


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ---------------------------------------------------------------------------
# Index maps
# ---------------------------------------------------------------------------
def pin_index_golden(ora):
    """Hand-written shard membership: S=16, N=2 contiguous / zig-zag ([CP] §2.1,
    [ZZ] §Zig Zag) and the page's own token-strided example with N=4, at S=16 and
    at S=12 (a multiple of N but not of 2N)."""
    for name, S, n in (("zigzag_S16_N2.txt", 16, 2), ("strided_S16_N4.txt", 16, 4),
                       ("strided_S12_N4.txt", 12, 4)):
        for line in _read_golden(name):
            head, toks = line.split(":")
            layout, r = head.split()
            want = [int(t) for t in toks.split()]
            got = ora.shard_members(S, n, layout)[int(r)]
            assert got == want, (layout, r, got, want)


def _closed_form_perm(S, N, layout):
    """Slot p -> global position, by the closed form of the 2N-chunk assignment:
    r = p div c, u = p mod c; g = r h + u if u < h else (2N-1-r) h + (u - h)."""
    if layout == "contiguous":
        return np.arange(S)
    if layout == "strided":  # slot p of shard r = p div c, offset u = p mod c: u N + r
        c = S // N
        return (np.arange(S) % c) * N + np.arange(S) // c
    c, h = S // N, S // (2 * N)
    p = np.arange(S)
    r, u = p // c, p % c
    return np.where(u < h, r * h + u, (2 * N - 1 - r) * h + (u - h))


def pin_index_bijection(ora):
    """perm is a bijection, inv o perm = id, contiguous is the identity, the
    loop-built zig-zag map equals the closed form, and every zig-zag shard holds
    early (< S/2) and late (>= S/2) tokens ([ZZ] §Zig Zag)."""
    for S, N in [(2, 1), (8, 1), (16, 2), (24, 3), (64, 4), (1024, 4), (96, 8), (128, 64)]:
        for layout in ("contiguous", "zigzag", "strided"):
            perm, inv = ora.index_maps(S, N, layout)
            assert sorted(perm.tolist()) == list(range(S))
            assert np.array_equal(inv[perm], np.arange(S))
            assert np.array_equal(perm[inv], np.arange(S))
            assert np.array_equal(perm, _closed_form_perm(S, N, layout)), (S, N, layout)
            if layout == "contiguous":
                assert np.array_equal(perm, np.arange(S))
            else:
                for shard in ora.shard_members(S, N, layout):
                    assert min(shard) < S // 2 <= max(shard)
            if layout == "strided":  # consecutive tokens land on consecutive shards
                assert all(inv[g] // (S // N) == g % N for g in range(S))


# ---------------------------------------------------------------------------
# Causal balance
# ---------------------------------------------------------------------------
def pin_balance(ora):
    """Causal pairs per shard: hand count, brute-force double loop, closed forms
    (contiguous c^2 r + c(c+1)/2, skewed; zig-zag h^2 (2N-1) + h(h+1), equal) and
    the C3 / C5 values."""
    for line in _read_golden("causal_pairs_S16_N2.txt"):
        layout, *vals = line.split()
        assert ora.causal_pairs_per_shard(16, 2, layout) == [int(x) for x in vals]
    for S, N in [(16, 2), (64, 4), (96, 3), (256, 8)]:
        for layout in ("contiguous", "zigzag", "strided"):
            got = ora.causal_pairs_per_shard(S, N, layout)
            members = ora.shard_members(S, N, layout)
            brute = []
            for shard in members:
                cnt = 0
                for i in shard:
                    for j in range(S):
                        if j <= i:
                            cnt += 1
                brute.append(cnt)
            assert got == brute
            assert sum(got) == S * (S + 1) // 2
    for S, N in [(65536, 8), (262144, 16)]:
        c, h = S // N, S // (2 * N)
        contig = ora.causal_pairs_per_shard(S, N, "contiguous")
        zz = ora.causal_pairs_per_shard(S, N, "zigzag")
        assert contig == [c * c * r + c * (c + 1) // 2 for r in range(N)]
        assert zz == [h * h * (2 * N - 1) + h * (h + 1)] * N
        # strided: shard r holds u N + r, u < c: sum of (u N + r + 1) = N c(c-1)/2 + c(r+1)
        assert ora.causal_pairs_per_shard(S, N, "strided") == [N * c * (c - 1) // 2 + c * (r + 1)
                                                                for r in range(N)]
    assert ora.causal_pairs_per_shard(65536, 8, "contiguous")[0] == 33_558_528
    assert ora.causal_pairs_per_shard(65536, 8, "contiguous")[7] == 503_320_576
    assert ora.causal_pairs_per_shard(65536, 8, "zigzag")[3] == 268_439_552
    assert ora.causal_pairs_per_shard(262144, 16, "contiguous")[0] == 134_225_920
    assert ora.causal_pairs_per_shard(262144, 16, "contiguous")[15] == 4_160_757_760
    assert ora.causal_pairs_per_shard(262144, 16, "zigzag")[9] == 2_147_491_840


# ---------------------------------------------------------------------------
# Forward by definition
# ---------------------------------------------------------------------------
def _torch_reference(q, k, v, causal, scale, slopes):
    """torch fp64 CPU: softmax(scale q k^T + bias + mask) v, and its autograd."""
    S = q.shape[2]
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = scale * torch.matmul(tq, tk.transpose(-1, -2))
    pos = torch.arange(S, dtype=torch.float64)
    if slopes is not None:
        dist = (pos[None, :] - pos[:, None]).abs()
        s = s - torch.tensor(slopes, dtype=torch.float64)[None, :, None, None] * dist
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(S, S, dtype=torch.bool), 1), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    o = torch.matmul(torch.softmax(s, dim=-1), tv)
    return tq, tk, tv, o, lse


def pin_torch_forward(ora):
    """One-shot torch fp64 softmax attention (a separate library routine)."""
    for (B, H, S, D), causal, alibi in itertools.product(
            [(1, 2, 37, 8), (2, 3, 64, 16)], [False, True], [False, True]):
        q, k, v = _qkv(B, H, S, D, 11 + S)
        scale = 1.0 / math.sqrt(D)
        sl = _slopes(H) if alibi else None
        _, _, _, o_t, l_t = _torch_reference(q, k, v, causal, scale, sl)
        o, l = ora.attention_forward(q, k, v, causal=causal, scale=scale, slopes=sl)
        assert np.max(np.abs(o - o_t.detach().numpy())) < 1e-12
        assert np.max(np.abs(l - l_t.detach().numpy())) < 1e-12


def _brute(q, k, v, causal, scale, slopes):
    """Pure-Python triple loop, written independently of the oracle."""
    B, H, S, D = q.shape
    O = np.zeros((B, H, S, D))
    L = np.zeros((B, H, S))
    for b in range(B):
        for h in range(H):
            for i in range(S):
                sc = []
                for j in range(S):
                    if causal and j > i:
                        continue
                    dot = 0.0
                    for d in range(D):
                        dot += q[b, h, i, d] * k[b, h, j, d]
                    val = dot * scale
                    if slopes is not None:
                        val -= slopes[h] * abs(i - j)
                    sc.append((j, val))
                mx = max(val for _, val in sc)
                tot = sum(math.exp(val - mx) for _, val in sc)
                L[b, h, i] = mx + math.log(tot)
                for j, val in sc:
                    w = math.exp(val - L[b, h, i])
                    for d in range(D):
                        O[b, h, i, d] += w * v[b, h, j, d]
    return O, L


def pin_brute_force(ora):
    for causal, alibi in itertools.product([False, True], [False, True]):
        q, k, v = _qkv(1, 2, 13, 4, 5)
        scale = 0.7
        sl = _slopes(2) if alibi else None
        ob, lb = _brute(q, k, v, causal, scale, sl)
        o, l = ora.attention_forward(q, k, v, causal=causal, scale=scale, slopes=sl)
        assert np.max(np.abs(o - ob)) < 1e-12 and np.max(np.abs(l - lb)) < 1e-12


def pin_rows_sum_to_one(ora):
    """softmax rows sum to 1: with V = 1 every output is exactly 1."""
    q, k, _ = _qkv(1, 2, 50, 8, 7)
    v = np.ones_like(q)
    for causal in (False, True):
        o, _ = ora.attention_forward(q, k, v, causal=causal, scale=0.5, slopes=_slopes(2))
        assert np.max(np.abs(o - 1.0)) < 1e-12


def pin_equal_keys(ora):
    """All keys equal: O_i = mean of V over the visible keys (causal: prefix mean)
    and LSE_i = scale q_i.k + ln(#visible)."""
    B, H, S, D = 1, 2, 40, 8
    q, _, v = _qkv(B, H, S, D, 9)
    kvec = _rng(3).standard_normal(D)
    k = np.broadcast_to(kvec, (B, H, S, D)).copy()
    scale = 0.3
    for causal in (False, True):
        o, l = ora.attention_forward(q, k, v, causal=causal, scale=scale)
        for i in range(S):
            n = i + 1 if causal else S
            want_o = v[:, :, :n].mean(axis=2)
            want_l = scale * (q[:, :, i] @ kvec) + math.log(n)
            assert np.max(np.abs(o[:, :, i] - want_o)) < 1e-12
            assert np.max(np.abs(l[:, :, i] - want_l)) < 1e-12


def pin_alibi_zero_query(ora):
    """Q = 0 with ALiBi: the row's LSE is a closed geometric series
    ([LC] §2.1.2 bias -|i-j| slope).  Causal: ln((1 - e^{-a(i+1)}) / (1 - e^{-a}));
    full: the two one-sided series around the diagonal."""
    B, H, S, D = 1, 4, 33, 4
    _, k, v = _qkv(B, H, S, D, 4)
    q = np.zeros((B, H, S, D))
    sl = _slopes(H)
    oc, lc = ora.attention_forward(q, k, v, causal=True, scale=0.25, slopes=sl)
    of, lf = ora.attention_forward(q, k, v, causal=False, scale=0.25, slopes=sl)
    for h in range(H):
        a = sl[h]
        g = lambda n: (1.0 - math.exp(-a * n)) / (1.0 - math.exp(-a))  # sum_{d<n} e^{-a d}
        for i in range(S):
            assert abs(lc[0, h, i] - math.log(g(i + 1))) < 1e-12
            assert abs(lf[0, h, i] - math.log(g(i + 1) + math.exp(-a) * g(S - 1 - i))) < 1e-12
            w = np.array([math.exp(-a * (i - j)) for j in range(i + 1)])
            want = (w[:, None] * v[0, h, :i + 1]).sum(axis=0) / w.sum()
            assert np.max(np.abs(oc[0, h, i] - want)) < 1e-12


def pin_shift_invariance(ora):
    """K <- K + c leaves O unchanged and shifts LSE_i by scale q_i.c;
    V <- V + c shifts O by c."""
    q, k, v = _qkv(1, 2, 30, 8, 12)
    cvec = _rng(8).standard_normal(8)
    scale = 0.4
    for causal in (False, True):
        o, l = ora.attention_forward(q, k, v, causal=causal, scale=scale, slopes=_slopes(2))
        o2, l2 = ora.attention_forward(q, k + cvec, v, causal=causal, scale=scale, slopes=_slopes(2))
        o3, _ = ora.attention_forward(q, k, v + cvec, causal=causal, scale=scale, slopes=_slopes(2))
        assert np.max(np.abs(o2 - o)) < 1e-11
        assert np.max(np.abs(l2 - (l + scale * (q @ cvec)))) < 1e-11
        assert np.max(np.abs(o3 - (o + cvec))) < 1e-11


# ---------------------------------------------------------------------------
# Ring-step merge and the online recurrence
# ---------------------------------------------------------------------------
def pin_merge_any_order(ora):
    """Keys split into random blocks; the blockwise LSE merge in any order equals
    the one-shot result ([ZZ] §Zig Zag: every Q meets every K/V block)."""
    r = _rng(21)
    B, H, S, D = 1, 2, 48, 8
    q, k, v = _qkv(B, H, S, D, 22)
    sl = _slopes(H)
    for causal in (False, True):
        o_ref, l_ref = ora.attention_forward(q, k, v, causal=causal, scale=0.35, slopes=sl)
        for _ in range(4):
            keys = r.permutation(S)
            cuts = np.sort(r.choice(np.arange(1, S), size=5, replace=False))
            blocks = np.split(keys, cuts)
            o = np.zeros((B, H, S, D))
            l = np.full((B, H, S), -np.inf)
            for blk in r.permutation(len(blocks)):
                ob, lb = ora.attention_forward(q, k, v, causal=causal, scale=0.35, slopes=sl,
                                               keys=np.sort(blocks[blk]))
                o, l = ora.lse_merge(o, l, ob, lb)
            assert np.max(np.abs(o - o_ref)) < 1e-12 and np.max(np.abs(l - l_ref)) < 1e-12
    # two empty partials merge to (O = 0, LSE = -inf)
    z = np.zeros((1, 3))
    om, lm = ora.lse_merge(z[..., None], np.full((1, 3), -np.inf), z[..., None] + 5.0,
                           np.full((1, 3), -np.inf))
    assert np.all(om == 0.0) and np.all(np.isneginf(lm))


def pin_ring_forward(ora):
    """Ring steps over N shards, both layouts, ring order and random visit
    orders: equal to one-shot attention in original order ([CP] §3.1)."""
    r = _rng(31)
    B, H, S, D = 1, 2, 48, 8
    q, k, v = _qkv(B, H, S, D, 32)
    sl = _slopes(H)
    for N, layout, causal in itertools.product([1, 2, 3], ["contiguous", "zigzag", "strided"], [False, True]):
        o_ref, l_ref = ora.attention_forward(q, k, v, causal=causal, scale=0.3, slopes=sl)
        o, l = ora.ring_forward(q, k, v, causal=causal, scale=0.3, slopes=sl, N=N, layout=layout)
        assert np.max(np.abs(o - o_ref)) < 1e-12 and np.max(np.abs(l - l_ref)) < 1e-12
        order = [r.permutation(N) for _ in range(N)]
        o, l = ora.ring_forward(q, k, v, causal=causal, scale=0.3, slopes=sl, N=N,
                                layout=layout, order=order)
        assert np.max(np.abs(o - o_ref)) < 1e-12 and np.max(np.abs(l - l_ref)) < 1e-12


def pin_online_recurrence(ora):
    """The running (m, l, O) recurrence ([LC] §3.1.2, corrected) equals one-shot."""
    q, k, v = _qkv(1, 2, 45, 8, 41)
    for causal, blk in itertools.product([False, True], [1, 7, 16, 64]):
        o_ref, l_ref = ora.attention_forward(q, k, v, causal=causal, scale=0.6, slopes=_slopes(2))
        o, l = ora.online_softmax_rows(q, k, v, causal=causal, scale=0.6, slopes=_slopes(2), block=blk)
        assert np.max(np.abs(o - o_ref)) < 1e-12 and np.max(np.abs(l - l_ref)) < 1e-12


# ---------------------------------------------------------------------------
# Backward
# ---------------------------------------------------------------------------
def pin_torch_backward(ora):
    """torch fp64 autograd of the one-shot forward."""
    for (B, H, S, D), causal, alibi in itertools.product(
            [(1, 2, 29, 8), (1, 1, 64, 16)], [False, True], [False, True]):
        q, k, v = _qkv(B, H, S, D, 51 + S)
        do = _rng(52).standard_normal((B, H, S, D))
        scale = 1.0 / math.sqrt(D)
        sl = _slopes(H) if alibi else None
        tq, tk, tv, o_t, _ = _torch_reference(q, k, v, causal, scale, sl)
        o_t.backward(torch.tensor(do))
        dq, dk, dv = ora.attention_backward(q, k, v, do, causal=causal, scale=scale, slopes=sl)
        assert np.max(np.abs(dq - tq.grad.numpy())) < 1e-11
        assert np.max(np.abs(dk - tk.grad.numpy())) < 1e-11
        assert np.max(np.abs(dv - tv.grad.numpy())) < 1e-11


def pin_backward_invariants(ora):
    """sum_j dV_j = sum_i dO_i (rows of P sum to 1); sum_j dK_j = 0 (rows of dS
    sum to 0); central finite differences of <O, dO>."""
    B, H, S, D = 1, 2, 20, 4
    q, k, v = _qkv(B, H, S, D, 61)
    do = _rng(62).standard_normal((B, H, S, D))
    sl = _slopes(H)
    for causal in (False, True):
        dq, dk, dv = ora.attention_backward(q, k, v, do, causal=causal, scale=0.5, slopes=sl)
        assert np.max(np.abs(dv.sum(axis=2) - do.sum(axis=2))) < 1e-11
        assert np.max(np.abs(dk.sum(axis=2))) < 1e-11

        def f(qq, kk, vv):
            o, _ = ora.attention_forward(qq, kk, vv, causal=causal, scale=0.5, slopes=sl)
            return float(np.sum(o * do))
        eps = 1e-5
        r = _rng(63)
        for name, grad in (("q", dq), ("k", dk), ("v", dv)):
            for _ in range(6):
                idx = (0, int(r.integers(H)), int(r.integers(S)), int(r.integers(D)))
                args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
                args[name][idx] += eps
                fp = f(args["q"], args["k"], args["v"])
                args[name][idx] -= 2 * eps
                fm = f(args["q"], args["k"], args["v"])
                fd = (fp - fm) / (2 * eps)
                assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def pin_backward_partial(ora):
    """dQ on a row subset and dK/dV on a key subset equal the full backward."""
    B, H, S, D = 1, 2, 40, 8
    q, k, v = _qkv(B, H, S, D, 71)
    do = _rng(72).standard_normal((B, H, S, D))
    sl = _slopes(H)
    for causal in (False, True):
        dq, dk, dv = ora.attention_backward(q, k, v, do, causal=causal, scale=0.45, slopes=sl)
        rows = np.array([0, 5, 17, 39])
        cols = np.array([3, 20, 33, 39])
        dqr = ora.backward_dq_rows(q, k, v, do, rows, causal=causal, scale=0.45, slopes=sl)
        dkc, dvc = ora.backward_dkdv_cols(q, k, v, do, cols, causal=causal, scale=0.45, slopes=sl)
        assert np.max(np.abs(dqr - dq[:, :, rows])) < 1e-12
        assert np.max(np.abs(dkc - dk[:, :, cols])) < 1e-12
        assert np.max(np.abs(dvc - dv[:, :, cols])) < 1e-12


# ---------------------------------------------------------------------------
# RoPE ([LC] §2.1.3)
# ---------------------------------------------------------------------------
def pin_rope_frequencies(ora):
    """theta_i = 1 / 10000^(2i/D): at D = 8 the four frequencies are 1, 1/10,
    1/100, 1/1000; at D = 128 the same values sit at i = 0, 16, 32, 48."""
    assert np.allclose(ora.rope_frequencies(8), [1.0, 0.1, 0.01, 0.001], rtol=1e-15, atol=0)
    f = ora.rope_frequencies(128)
    assert f.shape == (64,)
    assert np.allclose(f[[0, 16, 32, 48]], [1.0, 0.1, 0.01, 0.001], rtol=1e-15, atol=0)
    assert np.all(np.diff(f) < 0)


def pin_rope_unit_vectors(ora):
    """Closed form of the rotate-half formula on unit vectors, D = 8, with the
    frequencies written out: e_j (j < 4) goes to cos(t w_j) e_j + sin(t w_j) e_{j+4};
    e_{j+4} goes to -sin(t w_j) e_j + cos(t w_j) e_{j+4}."""
    w = [1.0, 0.1, 0.01, 0.001]
    pos = np.array([0, 1, 3, 7, 1000, 123457, 262143], dtype=np.float64)
    for j in range(8):
        x = np.zeros((len(pos), 8))
        x[:, j] = 1.0
        y = ora.rope_rotate(x, pos)
        i = j % 4
        want = np.zeros((len(pos), 8))
        for n, t in enumerate(pos):
            c, s = math.cos(t * w[i]), math.sin(t * w[i])
            if j < 4:
                want[n, i], want[n, i + 4] = c, s
            else:
                want[n, i], want[n, i + 4] = -s, c
        assert np.max(np.abs(y - want)) < 1e-9, (j, np.max(np.abs(y - want)))


def pin_rope_relative_position(ora):
    """The page's claim: the rotation encodes relative position.  The score
    <R(a) q, R(b) k> depends only on b - a: shifting both positions leaves it
    unchanged, and it equals <q, R(b - a) k>."""
    r = _rng(91)
    S, D = 40, 16
    q, k = r.standard_normal((S, D)), r.standard_normal((S, D))
    pos = r.integers(0, 5000, size=S).astype(np.float64)
    base = ora.rope_rotate(q, pos) @ ora.rope_rotate(k, pos).T
    for shift in (1.0, 37.0, 100000.0):
        got = ora.rope_rotate(q, pos + shift) @ ora.rope_rotate(k, pos + shift).T
        assert np.max(np.abs(got - base)) < 1e-9
    for a in range(0, S, 7):
        rel = ora.rope_rotate(k, pos - pos[a]) @ q[a]
        assert np.max(np.abs(rel - base[a])) < 1e-9


def pin_rope_orthogonal(ora):
    """A rotation: position 0 is the identity, each pair (i, i + D/2) keeps its
    length, the inverse undoes it, and rotations by a then b compose to a + b."""
    r = _rng(92)
    x = r.standard_normal((2, 3, 33, 64))
    pos = r.integers(0, 300000, size=33).astype(np.float64)
    assert np.array_equal(ora.rope_rotate(x, np.zeros(33)), x)
    y = ora.rope_rotate(x, pos)
    pair = lambda z: z[..., :32] ** 2 + z[..., 32:] ** 2  # noqa: E731
    assert np.max(np.abs(pair(y) - pair(x))) < 1e-10
    assert np.max(np.abs(ora.rope_rotate(y, pos, inverse=True) - x)) < 1e-10
    p2 = r.integers(0, 1000, size=33).astype(np.float64)
    assert np.max(np.abs(ora.rope_rotate(y, p2) - ora.rope_rotate(x, pos + p2))) < 1e-9
    # the inverse is the transpose: <R x, z> = <x, R^T z>
    z = r.standard_normal(x.shape)
    lhs = np.sum(y * z, axis=-1)
    rhs = np.sum(x * ora.rope_rotate(z, pos, inverse=True), axis=-1)
    assert np.max(np.abs(lhs - rhs)) < 1e-10


ALL_PINS = [
    pin_index_golden, pin_index_bijection, pin_balance, pin_torch_forward,
    pin_brute_force, pin_rows_sum_to_one, pin_equal_keys, pin_alibi_zero_query,
    pin_shift_invariance, pin_merge_any_order, pin_ring_forward,
    pin_online_recurrence, pin_torch_backward, pin_backward_invariants,
    pin_backward_partial, pin_rope_frequencies, pin_rope_unit_vectors,
    pin_rope_relative_position, pin_rope_orthogonal,
]
