"""Oracle for ring / zig-zag blockwise attention — TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg may
import this module.  The library never calls it, and it shares no code with the
CUDA path: it is a plain, slow fp64 restatement of what the method computes.

Pages cited (titles as printed):
  [CP]  "百万Token上下文训练的挑战与突破" (discosf.com news 4628517)
  [ZZ]  "大模型如何訓練百萬 Token 上下文：上下文并行與 Ring Attention" (Khang Pham)
  [LC]  "超长上下文技术" survey (intelliparadigm.com article 2061774)

What each function follows:
  shard_members / index_maps  [CP] §2.1 (contiguous split of the sequence into N
      equal pieces, one per device) and [ZZ] §Zig Zag Ring Attention (interleaved
      assignment so every device holds early and late tokens).  The interleaving
      used is the 2N-chunk form: the sequence is cut into 2N equal chunks and
      shard r holds chunk r followed by chunk 2N-1-r.  The token-strided form the
      same section prints (GPU 0 gets tokens 0, 4, 8, ..., GPU 1 gets 1, 5, 9, ...)
      is the third layout: shard r holds tokens r, r+N, r+2N, ...
  attention_forward           [LC] §2.1.2 (scores = q.k / sqrt(head dim), then the
      ALiBi bias -|i-j| * slope added) and [ZZ] §Zig Zag (causal: a token sees
      only earlier tokens; the diagonal is visible).  Plain softmax per query row
      over every visible key; LSE = natural-log log-sum-exp of the row.
  attention_backward          the analytic gradient of attention_forward (the pages
      name only the recompute strategy, [LC] §3.1.2): D_i = dO_i.O_i,
      dP = dO V^T, dS = P o (dP - D), dV = P^T dO, dQ = scale dS K, dK = scale dS^T Q.
  lse_merge / ring_forward    [ZZ] §Zig Zag (each shard's queries meet the K/V of
      every shard, one ring step at a time, until all pairs are covered) and
      [CP] §3.1 (device i receives the K/V of device i-1): step t pairs shard r
      with the K/V of shard (r - t) mod N; partial results are merged through
      their log-sum-exp.
  online_softmax_rows         [LC] §3.1.2 (running row max m and running sum l,
      output rescaled by exp(m_old - m_new)), in the corrected form where the
      block's own terms are also referred to the new maximum.

All arithmetic is float64.  Inputs are the exact stored values (fp32 or bf16)
upcast to float64, in ORIGINAL sequence order (index = global token position).

Every function here is pinned by the CPU tests in tests/test_oracle_pins.py
(closed forms, invariants, a brute-force triple loop, and torch fp64 autograd).
"""
from __future__ import annotations

import numpy as np

CONTIGUOUS = "contiguous"
ZIGZAG = "zigzag"
STRIDED = "strided"
LAYOUTS = (CONTIGUOUS, ZIGZAG, STRIDED)

# Rows of scores materialised at once: a memory bound only (each row's softmax
# is still taken over its whole key set in one go).
_ROW_ELEMS = 1 << 22


# ----------------------------------------------------------------------------
# Sequence -> shard assignment
# ----------------------------------------------------------------------------
def check_split(S: int, N: int, layout: str) -> None:
    if layout not in LAYOUTS:
        raise ValueError(f"unknown layout {layout!r}")
    if N < 1 or S < 0:
        raise ValueError("need N >= 1 and S >= 0")
    parts = 2 * N if layout == ZIGZAG else N  # 2N chunks; N equal pieces; tokens dealt out N at a time
    if S % parts:
        raise ValueError(f"S={S} is not divisible by {parts} ({layout}, N={N})")


def shard_members(S: int, N: int, layout: str) -> list[list[int]]:
    """Global token positions each shard holds, in the order the shard stores them.

    Built by walking the chunks one by one (no closed form), so that the tests can
    compare it with the closed-form maps of the library."""
    check_split(S, N, layout)
    shards: list[list[int]] = [[] for _ in range(N)]
    if layout == CONTIGUOUS:
        c = S // N
        for r in range(N):
            for u in range(c):
                shards[r].append(r * c + u)
    elif layout == STRIDED:
        for g in range(S):  # deal the tokens out to the shards in turn
            shards[g % N].append(g)
    else:
        h = S // (2 * N)
        chunks = [list(range(k * h, (k + 1) * h)) for k in range(2 * N)]
        for r in range(N):
            shards[r].extend(chunks[r])
            shards[r].extend(chunks[2 * N - 1 - r])
    return shards


def index_maps(S: int, N: int, layout: str):
    """perm[p] = global position stored at slot p of the shard-major buffer
    (the concatenation of the shards in order); inv[g] = slot of global position g."""
    members = shard_members(S, N, layout)
    perm = np.array([g for shard in members for g in shard], dtype=np.int64)
    inv = np.empty(S, dtype=np.int64)
    for p, g in enumerate(perm):
        inv[g] = p
    return perm, inv


def causal_pairs_per_shard(S: int, N: int, layout: str) -> list[int]:
    """Number of causally visible (query, key) pairs whose query a shard holds:
    a query at global position g sees keys 0..g, i.e. g + 1 of them."""
    return [int(sum(g + 1 for g in shard)) for shard in shard_members(S, N, layout)]


# ----------------------------------------------------------------------------
# Attention by definition
# ----------------------------------------------------------------------------
def _scores(qrows, kkeys, rows, keys, scale, slope, causal):
    """Scaled, biased, masked scores of query rows `rows` (vectors qrows) against
    keys `keys` (vectors kkeys, i.e. k[keys])."""
    s = scale * (qrows @ kkeys.T)
    if slope is not None:
        dist = np.abs(rows[:, None] - keys[None, :]).astype(np.float64)
        s = s - slope * dist
    if causal:
        s = np.where(keys[None, :] <= rows[:, None], s, -np.inf)
    return s


def _row_lse(s):
    """Natural-log log-sum-exp of each row; -inf for a row with no visible key."""
    m = s.max(axis=1)
    safe = np.where(np.isfinite(m), m, 0.0)
    tot = np.exp(s - safe[:, None]).sum(axis=1)
    with np.errstate(divide="ignore"):
        lse = safe + np.log(tot)
    return np.where(np.isfinite(m), lse, -np.inf)


def attention_forward(q, k, v, *, causal: bool, scale: float, slopes=None,
                      rows=None, keys=None):
    """Softmax attention by its definition.

    q, k, v: float64 [B, H, S, D] in original order.  rows: query positions to
    compute (default all); keys: the key positions taken into account (default
    all — a subset gives the partial result of one ring step).
    Returns O [B, H, R, D] and LSE [B, H, R] (natural log).  A row that sees no
    key gets O = 0 and LSE = -inf."""
    B, H, S, D = q.shape
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    keys = np.arange(S) if keys is None else np.asarray(keys, dtype=np.int64)
    R = len(rows)
    O = np.zeros((B, H, R, D))
    L = np.full((B, H, R), -np.inf)
    if R == 0 or len(keys) == 0:
        return O, L
    blk = max(1, _ROW_ELEMS // max(1, len(keys)))
    for b in range(B):
        for h in range(H):
            slope = None if slopes is None else float(slopes[h])
            kk, vk = k[b, h][keys], v[b, h][keys]
            for a in range(0, R, blk):
                r = rows[a:a + blk]
                s = _scores(q[b, h, r], kk, r, keys, scale, slope, causal)
                lse = _row_lse(s)
                p = np.exp(s - np.where(np.isfinite(lse), lse, 0.0)[:, None])
                p[~np.isfinite(lse)] = 0.0
                O[b, h, a:a + len(r)] = p @ vk
                L[b, h, a:a + len(r)] = lse
    return O, L


def attention_backward(q, k, v, dout, *, causal: bool, scale: float, slopes=None):
    """dQ, dK, dV of attention_forward (all rows, all keys) for the upstream
    gradient dout, from the recomputed probabilities P = exp(s - LSE)."""
    B, H, S, D = q.shape
    O, L = attention_forward(q, k, v, causal=causal, scale=scale, slopes=slopes)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    keys = np.arange(S)
    blk = max(1, _ROW_ELEMS // max(1, S))
    for b in range(B):
        for h in range(H):
            slope = None if slopes is None else float(slopes[h])
            Dvec = np.sum(dout[b, h] * O[b, h], axis=1)
            for a in range(0, S, blk):
                r = np.arange(a, min(S, a + blk))
                s = _scores(q[b, h, r], k[b, h], r, keys, scale, slope, causal)  # keys: all, in order
                lse = L[b, h, r]
                p = np.exp(s - lse[:, None])
                dp = dout[b, h, r] @ v[b, h].T
                ds = p * (dp - Dvec[r][:, None])
                dv[b, h] += p.T @ dout[b, h, r]
                dq[b, h, r] = scale * (ds @ k[b, h])
                dk[b, h] += scale * (ds.T @ q[b, h, r])
    return dq, dk, dv


def backward_dq_rows(q, k, v, dout, rows, *, causal: bool, scale: float, slopes=None):
    """dQ for the query positions `rows` only (each needs nothing but its own row)."""
    B, H, S, D = q.shape
    rows = np.asarray(rows, dtype=np.int64)
    O, L = attention_forward(q, k, v, causal=causal, scale=scale, slopes=slopes, rows=rows)
    keys = np.arange(S)
    dq = np.zeros((B, H, len(rows), D))
    for b in range(B):
        for h in range(H):
            slope = None if slopes is None else float(slopes[h])
            s = _scores(q[b, h, rows], k[b, h], rows, keys, scale, slope, causal)  # keys: all, in order
            p = np.exp(s - L[b, h][:, None])
            dp = dout[b, h, rows] @ v[b, h].T
            Dvec = np.sum(dout[b, h, rows] * O[b, h], axis=1)
            ds = p * (dp - Dvec[:, None])
            dq[b, h] = scale * (ds @ k[b, h])
    return dq


def backward_dkdv_cols(q, k, v, dout, cols, *, causal: bool, scale: float, slopes=None):
    """dK and dV for the key positions `cols` only.  Needs P and D for every query
    row that sees one of them, so the rows are recomputed in full."""
    B, H, S, D = q.shape
    cols = np.asarray(cols, dtype=np.int64)
    rows = np.arange(int(cols.min()), S) if causal else np.arange(S)
    O, L = attention_forward(q, k, v, causal=causal, scale=scale, slopes=slopes, rows=rows)
    dk = np.zeros((B, H, len(cols), D))
    dv = np.zeros((B, H, len(cols), D))
    blk = max(1, _ROW_ELEMS // max(1, len(cols)))
    for b in range(B):
        for h in range(H):
            slope = None if slopes is None else float(slopes[h])
            for a in range(0, len(rows), blk):
                r = rows[a:a + blk]
                s = _scores(q[b, h, r], k[b, h, cols], r, cols, scale, slope, causal)
                p = np.exp(s - L[b, h, a:a + len(r)][:, None])
                dp = dout[b, h, r] @ v[b, h, cols].T
                Dvec = np.sum(dout[b, h, r] * O[b, h, a:a + len(r)], axis=1)
                ds = p * (dp - Dvec[:, None])
                dv[b, h] += p.T @ dout[b, h, r]
                dk[b, h] += scale * (ds.T @ q[b, h, r])
    return dk, dv


# ----------------------------------------------------------------------------
# Ring-step form: partial results merged through their log-sum-exp
# ----------------------------------------------------------------------------
def lse_merge(o_a, lse_a, o_b, lse_b):
    """Merge two partial results over disjoint key sets:
    LSE = log(e^LSE_a + e^LSE_b), O = e^(LSE_a - LSE) O_a + e^(LSE_b - LSE) O_b.
    Two empty partials (-inf, -inf) merge to (-inf, 0)."""
    lse = np.logaddexp(lse_a, lse_b)
    fin = np.isfinite(lse)
    ref = np.where(fin, lse, 0.0)
    wa = np.where(fin, np.exp(lse_a - ref), 0.0)
    wb = np.where(fin, np.exp(lse_b - ref), 0.0)
    return wa[..., None] * o_a + wb[..., None] * o_b, lse


def ring_forward(q, k, v, *, causal: bool, scale: float, slopes=None, N: int,
                 layout: str, order=None):
    """Ring attention over N shards, returned in ORIGINAL order.

    Shard r's queries meet, at step t = 0..N-1, the keys of shard (r - t) mod N
    (or of order[r][t] when an explicit visit order is given); each step's partial
    (O_t, LSE_t) is merged into the running result with lse_merge."""
    B, H, S, D = q.shape
    members = shard_members(S, N, layout)
    O = np.zeros((B, H, S, D))
    L = np.full((B, H, S), -np.inf)
    for r in range(N):
        rows = np.array(members[r], dtype=np.int64)
        o_acc = np.zeros((B, H, len(rows), D))
        l_acc = np.full((B, H, len(rows)), -np.inf)
        steps = [(r - t) % N for t in range(N)] if order is None else list(order[r])
        for src in steps:
            keys = np.array(members[src], dtype=np.int64)
            o_t, l_t = attention_forward(q, k, v, causal=causal, scale=scale,
                                         slopes=slopes, rows=rows, keys=keys)
            o_acc, l_acc = lse_merge(o_acc, l_acc, o_t, l_t)
        O[:, :, rows] = o_acc
        L[:, :, rows] = l_acc
    return O, L


def online_softmax_rows(q, k, v, *, causal: bool, scale: float, slopes=None,
                        block: int = 64):
    """The running-(m, l, O) recurrence over key blocks for every query row:
    m_new = max(m, rowmax S_j); O = e^(m - m_new) O + e^(S_j - m_new) V_j;
    l = e^(m - m_new) l + rowsum e^(S_j - m_new); finally O / l and LSE = m + ln l."""
    B, H, S, D = q.shape
    rows = np.arange(S)
    O = np.zeros((B, H, S, D))
    L = np.full((B, H, S), -np.inf)
    for b in range(B):
        for h in range(H):
            slope = None if slopes is None else float(slopes[h])
            m = np.full(S, -np.inf)
            l = np.zeros(S)
            acc = np.zeros((S, D))
            for j0 in range(0, S, block):
                keys = np.arange(j0, min(S, j0 + block))
                s = _scores(q[b, h], k[b, h][keys], rows, keys, scale, slope, causal)
                m_new = np.maximum(m, s.max(axis=1))
                ref = np.where(np.isfinite(m_new), m_new, 0.0)
                alpha = np.where(np.isfinite(m), np.exp(m - ref), 0.0)
                p = np.exp(s - ref[:, None])
                acc = alpha[:, None] * acc + p @ v[b, h][keys]
                l = alpha * l + p.sum(axis=1)
                m = m_new
            with np.errstate(divide="ignore", invalid="ignore"):
                O[b, h] = np.where(l[:, None] > 0, acc / np.where(l > 0, l, 1.0)[:, None], 0.0)
                L[b, h] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return O, L
