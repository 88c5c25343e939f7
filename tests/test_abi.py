"""The C ABI on the host: the library loads, exports every declared entry point,
and the host-only calls and argument checks behave as include/ra.h states.
No kernel is launched here."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from context_ra_forward_gb300 import build, binding
    build.build()
    return binding.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "ra.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    assert L.ra_status_string(0) == b"RA_OK"
    assert L.ra_status_string(-5) == b"RA_ERR_TIMEOUT"
    assert L.ra_status_string(123) == b"RA_ERR_UNKNOWN"


@pytest.mark.parametrize("S,N,layout", [(16, 2, "zigzag"), (1024, 4, "zigzag"), (96, 3, "contiguous"),
                                        (65536, 8, "zigzag"), (24, 12, "zigzag"), (10, 1, "contiguous"),
                                        (16, 4, "strided"), (1200, 3, "strided"), (65536, 8, "strided")])
def test_index_map_matches_oracle_bit_exact(L, S, N, layout):
    from context_ra_forward_gb300 import binding
    perm, inv = binding.index_map(S, N, layout)
    operm, oinv = oracle.index_maps(S, N, layout)
    assert np.array_equal(perm, operm) and np.array_equal(inv, oinv)


def test_index_map_rejects(L):
    buf = np.empty(16, dtype=np.int64)
    assert L.ra_index_map(12, 4, 1, buf.ctypes.data, None) == -1   # 12 % 8 != 0
    assert L.ra_index_map(10, 3, 0, buf.ctypes.data, None) == -1
    assert L.ra_index_map(8, 0, 0, buf.ctypes.data, None) == -1
    assert L.ra_index_map(8, 2, 7, buf.ctypes.data, None) == -2
    assert L.ra_index_map(10, 4, 2, buf.ctypes.data, None) == -1   # strided: 10 % 4 != 0
    assert L.ra_index_map(0, 2, 1, None, None) == 0


def test_workspace_bytes(L):
    assert L.ra_backward_workspace_bytes(0, 1, 128, 128) == 0
    got = L.ra_backward_workspace_bytes(1, 2, 300, 64)
    rows = 600
    assert got == ((rows * 4 + 255) // 256) * 256 + ((rows * 64 * 4 + 255) // 256) * 256


def test_forward_path_and_validation(L):
    # argument checks run before any CUDA call, so they work without a GPU
    f = L.ra_forward_path
    assert f(1, 2, 1000, 96, 1, 4, 1) == -2       # D unsupported
    assert f(1, 2, 1000, 128, 1, 3, 1) == -1      # 1000 % 6
    assert f(1, 2, 1000, 128, 5, 4, 1) == -2      # dtype
    assert f(0, 2, 1024, 128, 1, 4, 1) == 0       # empty
    assert f(1, 2, 1024, 64, 0, 4, 1) == 2        # fp32 -> CUDA-core kernel
    fwd = L.ra_forward
    vp = ctypes.c_void_p(16)
    # zero-size problem: nothing to do, no launch, even with NULL pointers
    assert fwd(None, None, None, None, None, 1, 2, 0, 128, 1, 1, None, ctypes.c_float(0.0), 4, 1, None) == 0
    assert fwd(None, None, None, None, None, 1, 2, 64, 128, 1, 1, None, ctypes.c_float(0.0), 4, 1, None) == -1
    assert fwd(vp, vp, vp, ctypes.c_void_p(1 << 20), vp, 1, 2, 64, 100, 1, 1, None, ctypes.c_float(0.0), 4, 1, None) == -2
    mis = ctypes.c_void_p(8)
    assert fwd(mis, vp, vp, ctypes.c_void_p(1 << 20), vp, 1, 2, 64, 128, 1, 1, None, ctypes.c_float(0.0), 4, 1, None) == -3
    bp = L.ra_backward_path
    assert bp(1, 2, 1200, 128, 1, 3, 1) == 1      # 200-token chunks: tensor cores
    assert bp(1, 2, 1000, 128, 1, 4, 0) == 1      # contiguous, ragged tail
    assert bp(1, 2, 512, 128, 1, 4, 1) == 2       # 64-token chunks: CUDA cores
    assert bp(1, 2, 1024, 128, 0, 4, 1) == 2      # fp32
    assert bp(1, 2, 1024, 128, 2, 4, 1) == -2     # e4m3 has no backward
    assert bp(1, 2, 1000, 128, 1, 3, 1) == -1     # 1000 % 6
    # permute: aliasing input and output is rejected
    assert L.ra_zigzag_permute(vp, vp, 1, 1, 64, 128, 1, 4, 1, None) == -1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from context_ra_forward_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        binding.lib()


def _p(x):
    return ctypes.c_void_p(x)


F0 = ctypes.c_float(0.0)


def test_size_limits_rejected_before_launch(L):
    """The documented limits: S*D*e/16 < 2^31 per head and B*H*S*D < 4e18."""
    a, b, c, o = _p(1 << 20), _p(2 << 40), _p(3 << 40), _p(4 << 40)
    lse = _p(5 << 40)
    # S = 2^30 rows of D = 128 bf16: 2^34 16-byte chunks per head
    assert L.ra_forward(a, b, c, o, lse, 1, 1, 1 << 30, 128, 1, 1, None, F0, 1, 0, None) == -2
    assert L.ra_forward_path(1 << 20, 1 << 20, 1 << 20, 128, 1, 1, 0) == -2
    assert L.ra_zigzag_permute(a, o, 1, 1, 1 << 30, 128, 1, 1, 0, None) == -2


def test_rope_validation(L):
    x, y = _p(1 << 20), _p(1 << 40)
    rp = L.ra_rope_permute
    assert rp(x, y, 1, 2, 64, 128, 1, 4, 1, 1.0, 0, None) == -1            # base must exceed 1
    assert rp(x, y, 1, 2, 64, 128, 1, 4, 1, float("nan"), 0, None) == -1
    assert rp(x, y, 1, 2, 64, 128, 1, 4, 1, 10000.0, -1, None) == -1       # negative position offset
    assert rp(x, y, 1, 2, 64, 128, 1, 4, 1, 10000.0, (1 << 31) - 10, None) == -1  # past 2^31
    assert rp(x, y, 1, 2, 64, 128, 2, 4, 1, 10000.0, 0, None) == -2        # e4m3
    assert rp(x, y, 1, 2, 64, 96, 1, 4, 1, 10000.0, 0, None) == -2         # D
    assert rp(None, None, 1, 2, 0, 128, 1, 4, 1, 10000.0, 0, None) == 0    # empty: no launch
    assert rp(x, x, 1, 2, 64, 128, 1, 4, 1, 10000.0, 0, None) == -1        # in place
    assert rp(_p(8), y, 1, 2, 64, 128, 1, 4, 1, 10000.0, 0, None) == -3    # misaligned
    assert L.ra_rope_unpermute(x, y, 1, 2, 64, 128, 1, 4, 1, 0.5, 0, None) == -1


def test_fp8_ring_step_and_merge_validation(L):
    q, k, v, o, lse = (_p(n << 40) for n in range(1, 6))
    f8 = L.ra_forward_fp8
    one = ctypes.c_float(1.0)
    assert f8(q, k, v, ctypes.c_float(0.0), one, one, o, lse, 1, 2, 256, 128, 1, None, F0, 2, 1, None) == -1
    assert f8(q, k, v, one, ctypes.c_float(float("inf")), one, o, lse, 1, 2, 256, 128, 1, None, F0, 2, 1,
              None) == -1
    assert f8(q, k, v, one, one, one, o, lse, 1, 2, 256, 64, 1, None, F0, 2, 1, None) == -2  # D = 64
    rs = L.ra_forward_ring_step
    assert rs(q, k, v, o, lse, 1, 2, 2048, 128, 1, 1, None, F0, 4, 1, 4, None) == -1  # step == N
    assert rs(q, k, v, o, lse, 1, 2, 2048, 128, 1, 1, None, F0, 4, 1, -1, None) == -1
    assert rs(q, k, v, o, lse, 1, 2, 1024, 128, 1, 1, None, F0, 4, 1, 0, None) == -2  # runs of 128 rows
    mg = L.ra_lse_merge
    assert mg(q, k, v, o, None, 1, 1, 2, 64, 96, None) == -2              # D
    assert mg(q, k, v, o, lse, 2, 1, 2, 64, 128, None) == -2              # e4m3 output
    assert mg(None, None, None, None, None, 1, 1, 2, 0, 128, None) == 0   # empty
    assert mg(q, k, q, o, None, 1, 1, 2, 64, 128, None) == -1             # accumulator aliases the partial


def test_backward_validation(L):
    ptrs = [_p(n << 40) for n in range(1, 10)]  # q k v o lse do dq dk dv
    q, k, v, o, lse, do, dq, dk, dv = ptrs
    bw = L.ra_backward
    need = L.ra_backward_workspace_bytes(1, 2, 1024, 128)
    ws = _p(20 << 40)
    args = (1, 2, 1024, 128, 1, 1, None, F0, 4, 1, None)
    assert bw(q, k, v, o, lse, do, dq, dk, dv, ws, need - 1, *args) == -6       # workspace too small
    assert bw(q, k, v, o, lse, do, dq, dk, dv, None, need, *args) == -6
    assert bw(q, k, v, o, lse, do, dq, dk, dv, _p((20 << 40) + 16), need, *args) == -3  # not 256-aligned
    assert bw(q, k, v, o, lse, do, q, dk, dv, ws, need, *args) == -1            # dQ over Q
    assert bw(q, k, v, o, lse, do, dq, dk, dk, ws, need, *args) == -1           # dK over dV
    assert bw(q, k, v, o, lse, do, dq, dk, dv, ws, need, 1, 2, 1024, 128, 2, 1, None, F0, 4, 1, None) == -2


def test_noalloc_backward_validation_matches_backward(L):
    """ra_backward_noalloc answers an invalid call with the error ra_backward gives
    for it, even when the problem is also too large for its scratch buffer; only a
    valid problem beyond the buffer gets RA_ERR_WORKSPACE.  No CUDA call is made."""
    q, k, v, o, lse, do, dq, dk, dv = (_p(n << 40) for n in range(1, 10))
    nb = L.ra_backward_noalloc
    big = (1, 64, 65536)   # needs ~2 GB of scratch
    # (D, dtype, N, layout, scale) -> the error ra_backward returns for the same call
    for D, dt, N, layout, scale, want in [(96, 1, 8, 1, F0, -2),      # D unsupported
                                          (128, 7, 8, 1, F0, -2),     # dtype unknown
                                          (128, 2, 8, 1, F0, -2),     # e4m3 (needs scales)
                                          (128, 1, 8, 9, F0, -2),     # layout unknown
                                          (128, 1, 0, 1, F0, -1),     # N < 1
                                          (128, 1, 3, 1, F0, -1),     # S % 2N
                                          (128, 1, 8, 1, ctypes.c_float(float("nan")), -1)]:
        args = (*big, D, dt, 1, None, scale, N, layout, None)
        assert nb(q, k, v, o, lse, do, dq, dk, dv, *args) == want, (D, dt, N, layout)
        ws = _p(20 << 40)
        assert L.ra_backward(q, k, v, o, lse, do, dq, dk, dv, ws, 1 << 40, *args) == want
    # NULL and misaligned pointers, as ra_backward
    assert nb(None, k, v, o, lse, do, dq, dk, dv, *big, 128, 1, 1, None, F0, 8, 1, None) == -1
    assert nb(_p(8), k, v, o, lse, do, dq, dk, dv, *big, 128, 1, 1, None, F0, 8, 1, None) == -3
    # a valid problem beyond the buffer
    assert nb(q, k, v, o, lse, do, dq, dk, dv, *big, 128, 1, 1, None, F0, 8, 1, None) == -6
    # an empty problem: nothing to do
    assert nb(None, None, None, None, None, None, None, None, None, 1, 2, 0, 128, 1, 1, None, F0, 8, 1,
              None) == 0


@pytest.mark.parametrize("S,N,layout,causal", [(1024, 4, "zigzag", True), (1024, 4, "contiguous", True),
                                               (1024, 4, "strided", True), (1200, 3, "zigzag", True),
                                               (1300, 4, "strided", True), (512, 2, "zigzag", False)])
def test_shard_work_pairs_match_oracle(L, S, N, layout, causal):
    """The library's per-shard pair counts (from its closed-form map) equal the
    oracle's (from its explicit chunk walk); the tiles cover every visible pair."""
    from context_ra_forward_gb300 import binding
    pairs, full, part = binding.shard_work(S, N, layout, causal)
    want = oracle.causal_pairs_per_shard(S, N, layout) if causal else [S * (S // N)] * N
    assert list(pairs) == list(want)
    assert (full * 128 * 128 + part * 128 * 128 >= pairs).all()


def test_shard_work_balance_at_the_workloads(L):
    """Per-head tile counts at the causal 64K-token and 256K-token workloads,
    worked out by hand: with 128-token tiles, query tile i sees i full key tiles
    and one diagonal.  Contiguous 8 x 8192: shard r holds query tiles 64r..64r+63,
    so sum_i i = 2016 for shard 0 and 30688 for shard 7.  Zig-zag 16 chunks of 4096:
    shard r holds tiles 32r.. and 32(15-r).., 16352 for every shard.  Zig-zag 32
    chunks of 8192 (N = 16): 131008 per shard.  The pair counts are the closed
    forms c^2 r + c(c+1)/2 (contiguous) and h^2 (2N-1) + h(h+1) (zig-zag)."""
    from context_ra_forward_gb300 import binding
    pairs, full, part = binding.shard_work(65536, 8, "contiguous", True)
    assert full[0] == 2016 and full[7] == 30688 and list(part) == [64] * 8
    assert list(pairs) == [8192 ** 2 * r + 8192 * 8193 // 2 for r in range(8)]
    pairs, full, part = binding.shard_work(65536, 8, "zigzag", True)
    assert list(full) == [16352] * 8 and list(part) == [64] * 8
    assert list(pairs) == [4096 ** 2 * 15 + 4096 * 4097] * 8
    pairs, full, part = binding.shard_work(262144, 16, "zigzag", True)
    assert list(full) == [131008] * 16 and list(part) == [128] * 16
    assert list(pairs) == [8192 ** 2 * 31 + 8192 * 8193] * 16
