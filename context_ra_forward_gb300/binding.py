"""Thin ctypes binding over the C ABI of include/ra.h.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libra.so.  PyTorch supplies device memory and the current stream.
If the library is not built (or fails to load) every call raises; there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libra.so")

RA_OK = 0
STATUS_NAMES = {0: "RA_OK", -1: "RA_ERR_INVALID_ARG", -2: "RA_ERR_UNSUPPORTED",
                -3: "RA_ERR_MISALIGNED", -4: "RA_ERR_CUDA", -5: "RA_ERR_TIMEOUT",
                -6: "RA_ERR_WORKSPACE"}
DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float8_e4m3fn: 2}
LAYOUTS = {"contiguous": 0, "zigzag": 1, "strided": 2}


class RAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed: {STATUS_NAMES.get(status, status)}")


_lib = None

_i64, _i32, _vp, _f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_float


def lib() -> ctypes.CDLL:
    """Load libra.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built: run context_ra_forward_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    perm = [_vp, _vp, _i64, _i64, _i64, _i64, _i32, _i32, _i32, _vp]
    L.ra_index_map.argtypes = [_i64, _i32, _i32, _vp, _vp]
    L.ra_shard_work.argtypes = [_i64, _i32, _i32, _i32, _vp, _vp, _vp]
    L.ra_shard_work.restype = ctypes.c_int32
    L.ra_zigzag_permute.argtypes = perm
    L.ra_unpermute.argtypes = perm
    rope = [_vp, _vp, _i64, _i64, _i64, _i64, _i32, _i32, _i32, ctypes.c_double, _i64, _vp]
    L.ra_rope_permute.argtypes = rope
    L.ra_rope_unpermute.argtypes = rope
    L.ra_forward.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32, _i32, _vp,
                             _f32, _i32, _i32, _vp]
    L.ra_backward_workspace_bytes.argtypes = [_i64, _i64, _i64, _i64]
    L.ra_backward_workspace_bytes.restype = ctypes.c_size_t
    L.ra_backward.argtypes = [_vp] * 10 + [ctypes.c_size_t, _i64, _i64, _i64, _i64, _i32, _i32,
                                           _vp, _f32, _i32, _i32, _vp]
    L.ra_status_string.argtypes = [_i32]
    L.ra_status_string.restype = ctypes.c_char_p
    L.ra_check_device_status.argtypes = [_vp, _vp]
    L.ra_forward_path.argtypes = [_i64, _i64, _i64, _i64, _i32, _i32, _i32]
    L.ra_backward_path.argtypes = [_i64, _i64, _i64, _i64, _i32, _i32, _i32]
    L.ra_backward_path.restype = ctypes.c_int32
    L.ra_debug_wait_timeout.argtypes = [_i32, _vp]
    L.ra_forward_fp8.argtypes = [_vp, _vp, _vp, _f32, _f32, _f32, _vp, _vp, _i64, _i64, _i64, _i64, _i32,
                                 _vp, _f32, _i32, _i32, _vp]
    L.ra_forward_fp8.restype = ctypes.c_int32
    L.ra_forward_ring_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32, _i32, _vp,
                                       _f32, _i32, _i32, _i32, _vp]
    L.ra_forward_ring_step.restype = ctypes.c_int32
    L.ra_lse_merge.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i64, _i64, _vp]
    L.ra_lse_merge.restype = ctypes.c_int32
    L.ra_debug_wait_sites.argtypes = [_vp, _i32]
    L.ra_debug_wait_sites.restype = ctypes.c_int32
    L.ra_last_cuda_error.argtypes = []
    L.ra_last_cuda_error.restype = ctypes.c_char_p
    L.ra_backward_noalloc.argtypes = [_vp] * 9 + [_i64, _i64, _i64, _i64, _i32, _i32, _vp, _f32, _i32,
                                                    _i32, _vp]
    L.ra_backward_noalloc.restype = ctypes.c_int32
    L.ra_noalloc_scratch_bytes.argtypes = []
    L.ra_noalloc_scratch_bytes.restype = ctypes.c_size_t
    L.ra_kernel_launch_count.argtypes = []
    L.ra_kernel_launch_count.restype = ctypes.c_int64
    for name in ("ra_index_map", "ra_zigzag_permute", "ra_unpermute", "ra_forward", "ra_backward",
                 "ra_check_device_status", "ra_forward_path", "ra_debug_wait_timeout"):
        getattr(L, name).restype = ctypes.c_int32
    _lib = L
    return L


def _check(status: int, what: str) -> None:
    if status != RA_OK:
        if status == -4:
            what = f"{what} [{lib().ra_last_cuda_error().decode()}]"
        raise RAError(status, what)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _bhsd(t: torch.Tensor, name: str):
    if t.dim() != 4:
        raise ValueError(f"{name} must be [B, H, S, D]")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if t.dtype not in DTYPES:
        raise ValueError(f"{name}: dtype {t.dtype} not supported (float32, bfloat16, float8_e4m3fn)")
    return t.shape


def _layout(layout: str) -> int:
    if layout not in LAYOUTS:
        raise ValueError(f"layout must be one of {sorted(LAYOUTS)}")
    return LAYOUTS[layout]


def index_map(S: int, N: int, layout: str):
    """(perm, inv) as int64 numpy arrays: perm[slot] = global position, inv = its inverse."""
    perm = np.empty(S, dtype=np.int64)
    inv = np.empty(S, dtype=np.int64)
    _check(lib().ra_index_map(S, N, _layout(layout), perm.ctypes.data, inv.ctypes.data), "ra_index_map")
    return perm, inv


def shard_work(S: int, N: int, layout: str, causal: bool = True):
    """Per shard, for one head: (visible pairs, fully visible 128x128 tiles,
    partially visible tiles), each an int64 numpy array of N entries."""
    pairs, full, part = (np.empty(N, dtype=np.int64) for _ in range(3))
    _check(lib().ra_shard_work(S, N, _layout(layout), int(bool(causal)), pairs.ctypes.data, full.ctypes.data,
                               part.ctypes.data), "ra_shard_work")
    return pairs, full, part


def _permute(fn, x, N, layout, out, stream):
    B, H, S, D = _bhsd(x, "x")
    y = torch.empty_like(x) if out is None else out
    _bhsd(y, "out")
    _check(fn(_ptr(x), _ptr(y), B, H, S, D, DTYPES[x.dtype], N, _layout(layout), _stream(stream)),
           fn.__name__)
    return y


def zigzag_permute(x, N: int, layout: str = "zigzag", out=None, stream=None):
    """Original order -> shard-major order (ra_zigzag_permute)."""
    return _permute(lib().ra_zigzag_permute, x, N, layout, out, stream)


def unpermute(x, N: int, layout: str = "zigzag", out=None, stream=None):
    """Shard-major order -> original order (ra_unpermute)."""
    return _permute(lib().ra_unpermute, x, N, layout, out, stream)


def _rope(fn, x, N, layout, base, pos0, out, stream):
    B, H, S, D = _bhsd(x, "x")
    y = torch.empty_like(x) if out is None else out
    _bhsd(y, "out")
    if y.shape != x.shape or y.dtype != x.dtype:
        raise ValueError("out must match x in shape and dtype")
    _check(fn(_ptr(x), _ptr(y), B, H, S, D, DTYPES[x.dtype], N, _layout(layout), float(base), int(pos0),
              _stream(stream)), fn.__name__)
    return y


def rope_permute(x, N: int, layout: str = "zigzag", *, base: float = 10000.0, pos0: int = 0, out=None,
                 stream=None):
    """RoPE at each row's global position, fused with original -> shard-major (ra_rope_permute)."""
    return _rope(lib().ra_rope_permute, x, N, layout, base, pos0, out, stream)


def rope_unpermute(x, N: int, layout: str = "zigzag", *, base: float = 10000.0, pos0: int = 0, out=None,
                   stream=None):
    """The transpose: shard-major -> original with the inverse rotation (ra_rope_unpermute)."""
    return _rope(lib().ra_rope_unpermute, x, N, layout, base, pos0, out, stream)


def forward_path(B, H, S, D, dtype, N, layout) -> int:
    """1 = tensor-core kernel, 2 = CUDA-core fp32 kernel, 0 = empty, < 0 = rejected."""
    return lib().ra_forward_path(B, H, S, D, DTYPES[dtype], N, _layout(layout))


def backward_path(B, H, S, D, dtype, N, layout) -> int:
    """The kernel ra_backward runs (16-byte aligned LSE): 1 = tensor-core, 2 = CUDA-core
    fp32, 0 = empty, < 0 = rejected."""
    return lib().ra_backward_path(B, H, S, D, DTYPES[dtype], N, _layout(layout))


def forward(q, k, v, *, causal=False, alibi_slopes=None, softmax_scale=None, N=1,
            layout="contiguous", out=None, lse=None, stream=None):
    """Exact attention over N virtual ring shards (ra_forward).  q/k/v are
    [B, H, S, D] in shard-major order; returns (o, lse) in the same order."""
    B, H, S, D = _bhsd(q, "q")
    for t, n in ((k, "k"), (v, "v")):
        if _bhsd(t, n) != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{n} must match q in shape and dtype")
    o = torch.empty_like(q) if out is None else out
    lse_t = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    if alibi_slopes is not None:
        if alibi_slopes.dtype != torch.float32 or not alibi_slopes.is_cuda or alibi_slopes.numel() != H:
            raise ValueError("alibi_slopes must be a float32 CUDA tensor of H elements")
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check(lib().ra_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse_t), B, H, S, D,
                            DTYPES[q.dtype], int(bool(causal)), _ptr(alibi_slopes), scale, N,
                            _layout(layout), _stream(stream)), "ra_forward")
    return o, lse_t


def backward_workspace_bytes(B, H, S, D) -> int:
    return int(lib().ra_backward_workspace_bytes(B, H, S, D))


def backward(q, k, v, o, lse, dout, *, causal=False, alibi_slopes=None, softmax_scale=None,
             N=1, layout="contiguous", workspace=None, out=None, stream=None):
    """dQ, dK, dV (ra_backward), recomputing probabilities from the saved LSE."""
    B, H, S, D = _bhsd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        if _bhsd(t, n) != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{n} must match q in shape and dtype")
    need = backward_workspace_bytes(B, H, S, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    dq, dk, dv = out if out is not None else (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check(lib().ra_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                             _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), B, H, S, D,
                             DTYPES[q.dtype], int(bool(causal)), _ptr(alibi_slopes), scale, N,
                             _layout(layout), _stream(stream)), "ra_backward")
    return dq, dk, dv


def check_device_status(stream=None):
    """Synchronise and read/clear the device status word: (status, [code, kernel, block, site])."""
    detail = (ctypes.c_int32 * 4)()
    st = lib().ra_check_device_status(_stream(stream), ctypes.cast(detail, ctypes.c_void_p))
    return st, list(detail)


def debug_wait_timeout(limit_us: int, stream=None) -> None:
    _check(lib().ra_debug_wait_timeout(limit_us, _stream(stream)), "ra_debug_wait_timeout")


def kernel_launch_count() -> int:
    """Kernels the library has launched in this process (host-side counter)."""
    return int(lib().ra_kernel_launch_count())


def backward_noalloc(q, k, v, o, lse, dout, *, causal=False, alibi_slopes=None, softmax_scale=None,
                     N=1, layout="contiguous", out=None, stream=None):
    """dQ, dK, dV through ra_backward_noalloc: the same backward, for callers that
    cannot allocate device memory at this point (a framework that owns every
    allocation, memory fixed at start-up, a loop that cannot take an allocation's
    synchronisation).  The library's own fixed scratch buffer replaces the
    workspace, so problems larger than it are rejected.  The outputs here are
    allocated by torch unless `out` supplies them."""
    B, H, S, D = _bhsd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        if _bhsd(t, n) != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{n} must match q in shape and dtype")
    dq, dk, dv = out if out is not None else (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check(lib().ra_backward_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                                     _ptr(dk), _ptr(dv), B, H, S, D, DTYPES[q.dtype], int(bool(causal)),
                                     _ptr(alibi_slopes), scale, N, _layout(layout), _stream(stream)),
           "ra_backward_noalloc")
    return dq, dk, dv


def noalloc_scratch_bytes() -> int:
    return int(lib().ra_noalloc_scratch_bytes())


def debug_wait_sites():
    """Per warp of the first failing block: (site, parity, barrier address low bits)
    of the wait that gave up, or None for warps that did not give up."""
    n = lib().ra_debug_wait_sites(None, 0)
    buf = (ctypes.c_int32 * n)()
    lib().ra_debug_wait_sites(ctypes.cast(buf, ctypes.c_void_p), n)
    return [None if v == 0 else ((v >> 24) & 0xff, (v >> 16) & 1, v & 0xffff) for v in buf]


def forward_ring_step(q, k, v, step, *, causal=False, alibi_slopes=None, softmax_scale=None, N=1,
                      layout="contiguous", out=None, lse=None, stream=None):
    """One ring step as a separate partial (ra_forward_ring_step): returns fp32
    (o_step, lse_step) for the queries of every shard r against the K/V of shard
    (r - step) mod N."""
    B, H, S, D = _bhsd(q, "q")
    for t, n in ((k, "k"), (v, "v")):
        if _bhsd(t, n) != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{n} must match q in shape and dtype")
    o = torch.empty((B, H, S, D), dtype=torch.float32, device=q.device) if out is None else out
    lse_t = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check(lib().ra_forward_ring_step(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse_t), B, H, S, D,
                                      DTYPES[q.dtype], int(bool(causal)), _ptr(alibi_slopes), scale, N,
                                      _layout(layout), int(step), _stream(stream)), "ra_forward_ring_step")
    return o, lse_t


def lse_merge(o_acc, lse_acc, o_step, lse_step, out=None, stream=None):
    """Merge a ring-step partial into the accumulated one in place (ra_lse_merge);
    `out` (fp32 or bf16, optional) also receives the merged O."""
    B, H, S, D = o_acc.shape
    for t, n in ((o_acc, "o_acc"), (o_step, "o_step")):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.shape != o_acc.shape:
            raise ValueError(f"{n} must be a contiguous fp32 CUDA tensor [B, H, S, D]")
    out_dt = DTYPES[out.dtype] if out is not None else 0
    _check(lib().ra_lse_merge(_ptr(o_acc), _ptr(lse_acc), _ptr(o_step), _ptr(lse_step), _ptr(out), out_dt,
                              B, H, S, D, _stream(stream)), "ra_lse_merge")
    return o_acc, lse_acc


def forward_fp8(q, k, v, q_scale, k_scale, v_scale, *, causal=False, alibi_slopes=None, softmax_scale=None,
                N=1, layout="contiguous", out=None, lse=None, stream=None):
    """ra_forward_fp8: e4m3 q/k/v (torch.float8_e4m3fn, shard-major) with per-tensor
    scales; returns (o bf16, lse fp32)."""
    B, H, S, D = _bhsd(q, "q")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if _bhsd(t, n) != q.shape or t.dtype != torch.float8_e4m3fn:
            raise ValueError(f"{n} must be float8_e4m3fn and match q in shape")
    o = torch.empty((B, H, S, D), dtype=torch.bfloat16, device=q.device) if out is None else out
    lse_t = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check(lib().ra_forward_fp8(_ptr(q), _ptr(k), _ptr(v), float(q_scale), float(k_scale), float(v_scale),
                                _ptr(o), _ptr(lse_t), B, H, S, D, int(bool(causal)), _ptr(alibi_slopes), scale,
                                N, _layout(layout), _stream(stream)), "ra_forward_fp8")
    return o, lse_t
