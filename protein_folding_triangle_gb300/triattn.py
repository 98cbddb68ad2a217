"""Python binding of libtriattn (ctypes; argument marshalling only).

Every step of the computation runs in the CUDA kernels behind the C ABI in
``include/triattn.h``.  This module only checks tensor dtypes and shapes,
allocates outputs with torch (device memory), passes raw pointers and the
current CUDA stream, and raises on a non-OK status.  There is no fallback:
if the shared library is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

_LIB = None
_LOCK = threading.Lock()

STATUS = {
    0: "TRIATTN_OK",
    1: "TRIATTN_ERR_INVALID_ARG",
    2: "TRIATTN_ERR_UNSUPPORTED",
    3: "TRIATTN_ERR_WORKSPACE",
    4: "TRIATTN_ERR_CUDA",
    5: "TRIATTN_ERR_TIMEOUT",
}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(6)

EXPORTED = ("triattn_status_string", "triattn_fwd_workspace_bytes", "triattn_bwd_workspace_bytes", "tri_attn_fwd",
            "tri_attn_bwd",
            "triattn_device_status", "triattn_set_wait_limit_ns", "triattn_trace_enable", "triattn_trace_read",
            "triattn_test_set_starve", "tri_attn_bwd_noalloc", "triattn_bwd_atomic_workspace_bytes",
            "tri_attn_bwd_atomic_ablation", "tri_attn_dbias_combine", "triattn_module_ctx_bytes",
            "triattn_module_workspace_bytes", "tri_attn_module_fwd", "tri_attn_module_bwd",
            "triattn_trimul_ctx_bytes", "triattn_trimul_workspace_bytes", "triattn_trimul_fwd",
            "triattn_trimul_bwd", "triattn_gemm_workspace_bytes", "triattn_gemm", "tri_attn_fwd_strided",
            "tri_attn_bwd_strided")

FLAG_DBIAS_FP32 = 1

NOALLOC_SCRATCH_BYTES = 64 << 20


class TraceEntry(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_char_p), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double),
                ("min_ms", ctypes.c_double), ("max_ms", ctypes.c_double)]


class TriAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("N_o", ctypes.c_int), ("N", ctypes.c_int), ("H", ctypes.c_int),
                ("D", ctypes.c_int), ("flags", ctypes.c_uint)]


class Layout(ctypes.Structure):
    """triattn_layout: row (b, o, h, n) of a [B, N_o, H, N, D] tensor starts
    slice * (b N_o + o) + head * h + row * n elements from its base."""
    _fields_ = [("slice", ctypes.c_longlong), ("head", ctypes.c_longlong), ("row", ctypes.c_longlong)]


class ModuleShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("N", ctypes.c_int), ("C", ctypes.c_int), ("H", ctypes.c_int),
                ("D", ctypes.c_int), ("flags", ctypes.c_uint)]


class TriMulShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("N", ctypes.c_int), ("C_z", ctypes.c_int), ("C_h", ctypes.c_int),
                ("direction", ctypes.c_int), ("flags", ctypes.c_uint)]


TRIMUL_DIRECTIONS = {"outgoing": 0, "incoming": 1}


def _declare(lib):
    vp, sp = ctypes.c_void_p, ctypes.POINTER(Shape)
    lib.triattn_status_string.argtypes = [ctypes.c_int]
    lib.triattn_status_string.restype = ctypes.c_char_p
    lib.triattn_bwd_workspace_bytes.argtypes = [sp]
    lib.triattn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.triattn_fwd_workspace_bytes.argtypes = [sp]
    lib.triattn_fwd_workspace_bytes.restype = ctypes.c_size_t
    lib.tri_attn_fwd.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.tri_attn_fwd.restype = ctypes.c_int
    lib.tri_attn_bwd.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lp = ctypes.POINTER(Layout)
    lib.tri_attn_fwd_strided.argtypes = [sp, vp, vp, vp, lp, vp, vp, vp, vp, vp, lp, vp, ctypes.c_size_t, vp]
    lib.tri_attn_fwd_strided.restype = ctypes.c_int
    lib.tri_attn_bwd_strided.argtypes = ([sp, vp, vp, vp, lp, vp, vp, vp, vp, lp, vp, vp, lp, vp, vp, vp, lp, vp, vp,
                                          ctypes.c_size_t, vp])
    lib.tri_attn_bwd_strided.restype = ctypes.c_int
    lib.tri_attn_bwd.restype = ctypes.c_int
    lib.triattn_device_status.argtypes = [vp]
    lib.triattn_device_status.restype = ctypes.c_int
    lib.triattn_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.triattn_set_wait_limit_ns.restype = None
    lib.triattn_trace_enable.argtypes = [ctypes.c_int]
    lib.triattn_trace_enable.restype = None
    lib.triattn_trace_read.argtypes = [ctypes.POINTER(TraceEntry), ctypes.c_int]
    lib.triattn_trace_read.restype = ctypes.c_int
    lib.triattn_test_set_starve.argtypes = [ctypes.c_int]
    lib.triattn_test_set_starve.restype = None
    lib.tri_attn_bwd_noalloc.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.tri_attn_bwd_noalloc.restype = ctypes.c_int
    lib.triattn_bwd_atomic_workspace_bytes.argtypes = [sp, ctypes.c_int]
    lib.triattn_bwd_atomic_workspace_bytes.restype = ctypes.c_size_t
    lib.tri_attn_bwd_atomic_ablation.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                                 vp, ctypes.c_size_t, vp]
    lib.tri_attn_bwd_atomic_ablation.restype = ctypes.c_int
    lib.tri_attn_dbias_combine.argtypes = [sp, vp, ctypes.c_int, vp, vp]
    lib.tri_attn_dbias_combine.restype = ctypes.c_int
    mp = ctypes.POINTER(ModuleShape)
    lib.triattn_module_ctx_bytes.argtypes = [mp]
    lib.triattn_module_ctx_bytes.restype = ctypes.c_size_t
    lib.triattn_module_workspace_bytes.argtypes = [mp]
    lib.triattn_module_workspace_bytes.restype = ctypes.c_size_t
    lib.tri_attn_module_fwd.argtypes = [mp] + [vp] * 9 + [ctypes.c_size_t, vp]
    lib.tri_attn_module_fwd.restype = ctypes.c_int
    lib.tri_attn_module_bwd.argtypes = [mp] + [vp] * 13 + [ctypes.c_size_t, vp]
    lib.tri_attn_module_bwd.restype = ctypes.c_int
    tp = ctypes.POINTER(TriMulShape)
    lib.triattn_trimul_ctx_bytes.argtypes = [tp]
    lib.triattn_trimul_ctx_bytes.restype = ctypes.c_size_t
    lib.triattn_trimul_workspace_bytes.argtypes = [tp]
    lib.triattn_trimul_workspace_bytes.restype = ctypes.c_size_t
    lib.triattn_trimul_fwd.argtypes = [tp] + [vp] * 11 + [ctypes.c_size_t, vp]
    lib.triattn_trimul_fwd.restype = ctypes.c_int
    lib.triattn_trimul_bwd.argtypes = [tp] + [vp] * 16 + [ctypes.c_size_t, vp]
    lib.triattn_trimul_bwd.restype = ctypes.c_int
    ll = ctypes.c_longlong
    lib.triattn_gemm_workspace_bytes.argtypes = [ctypes.c_int] * 4
    lib.triattn_gemm_workspace_bytes.restype = ctypes.c_size_t
    lib.triattn_gemm.argtypes = ([ctypes.c_int] * 5 + [vp, ll, vp, ll, vp, ll, ctypes.c_int, ctypes.c_int, ll, ll, ll,
                                 vp, ctypes.c_size_t, vp])
    lib.triattn_gemm.restype = ctypes.c_int
    return lib


def library_path() -> str:
    return _build.lib_path()


def load(path: Optional[str] = None):
    """Load libtriattn (built in-tree by ``build.build()``); raises if absent."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            p = path or library_path()
            if not os.path.exists(p):
                raise RuntimeError(f"libtriattn is not built ({p} missing): run __graft_entry__.build()")
            _LIB = _declare(ctypes.CDLL(p))
    return _LIB


def shape_of(q: torch.Tensor) -> Shape:
    if q.dim() != 5:
        raise ValueError("q must be [B, N_o, H, N, D]")
    B, No, H, N, D = q.shape
    return Shape(B, No, N, H, D, 0)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(t: torch.Tensor, name: str, shape, dtype=torch.bfloat16):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _raise(code: int, where: str):
    if code != OK:
        raise TriAttnError(code, where)


def bwd_workspace_bytes(q_or_shape) -> int:
    s = q_or_shape if isinstance(q_or_shape, Shape) else shape_of(q_or_shape)
    return int(load().triattn_bwd_workspace_bytes(ctypes.byref(s)))


def fwd_workspace_bytes(q_or_shape) -> int:
    s = q_or_shape if isinstance(q_or_shape, Shape) else shape_of(q_or_shape)
    return int(load().triattn_fwd_workspace_bytes(ctypes.byref(s)))


def tri_attn_fwd(q, k, v, bias, mask=None, *, save_residual: bool = True, out=None, workspace=None, stream=None):
    """Forward.  Returns (o [B,N_o,H,N,D] bf16, lse [B,N_o,H,N] fp32,
    o_resid bf16 or None).  ``out`` may pass preallocated (o, lse, o_resid),
    ``workspace`` a uint8 device buffer of ``fwd_workspace_bytes`` bytes
    (allocated per call otherwise)."""
    s = shape_of(q)
    B, No, H, N, D = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, (B, No, H, N, D))
    _check(bias, "bias", (B, H, N, N))
    if mask is not None:
        _check(mask, "mask", (B, No, N))
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty((B, No, H, N), dtype=torch.float32, device=q.device)
        resid = torch.empty_like(q) if save_residual else None
    else:
        o, lse, resid = out
    if workspace is None:
        need = fwd_workspace_bytes(s)
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device) if need > 0 else None
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = load().tri_attn_fwd(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(mask), _ptr(o),
                               _ptr(lse), _ptr(resid), _ptr(workspace), ctypes.c_size_t(nbytes), _stream_ptr(stream))
    _raise(code, "tri_attn_fwd")
    return o, lse, resid


def tri_attn_bwd(q, k, v, bias, mask, o, o_resid, lse, do, *, workspace=None, out=None, stream=None,
                 dbias_fp32: bool = False):
    """Backward.  ``o_resid=None`` turns the residual compensation off.
    Returns (dq, dk, dv, dbias) in bf16; with ``dbias_fp32`` dbias is the FP32
    sum over this call's outer slices (a shard's part, see tri_attn_dbias_combine)."""
    s = shape_of(q)
    if dbias_fp32:
        s.flags = FLAG_DBIAS_FP32
    B, No, H, N, D = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check(t, name, (B, No, H, N, D))
    if o_resid is not None:
        _check(o_resid, "o_resid", (B, No, H, N, D))
    _check(bias, "bias", (B, H, N, N))
    _check(lse, "lse", (B, No, H, N), torch.float32)
    if mask is not None:
        _check(mask, "mask", (B, No, N))
    need = bwd_workspace_bytes(s)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        dbias = torch.empty(bias.shape, dtype=torch.float32 if dbias_fp32 else torch.bfloat16, device=q.device)
    else:
        dq, dk, dv, dbias = out
    _check(dbias, "dbias", tuple(bias.shape), torch.float32 if dbias_fp32 else torch.bfloat16)
    code = load().tri_attn_bwd(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(mask), _ptr(o),
                               _ptr(o_resid), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias),
                               _ptr(workspace), ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                               _stream_ptr(stream))
    _raise(code, "tri_attn_bwd")
    return dq, dk, dv, dbias


def layout_of(t: torch.Tensor) -> Layout:
    """The row layout of a [B, N_o, H, N, D] view whose D features are
    contiguous and whose b stride is N_o times its o stride (e.g. the heads of
    pair rows: ``P.view(B, N, N, ld)[..., c:c + H*D].unflatten(-1, (H, D))
    .permute(0, 1, 3, 2, 4)``)."""
    if t.dim() != 5 or t.stride(4) != 1:
        raise ValueError("expected a [B, N_o, H, N, D] view with contiguous features")
    if t.shape[0] > 1 and t.stride(0) != t.shape[1] * t.stride(1):
        raise ValueError("the b stride must be N_o times the o stride")
    return Layout(t.stride(1), t.stride(2), t.stride(3))


def _check_view(t, name, shape, lay: Layout):
    if t is None or not t.is_cuda or t.dtype != torch.bfloat16 or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be a bf16 CUDA view of shape {tuple(shape)}")
    got = layout_of(t)
    if (got.slice, got.head, got.row) != (lay.slice, lay.head, lay.row):
        raise ValueError(f"{name} does not share the layout of its group")


def tri_attn_fwd_strided(q, k, v, bias, mask, o, lse, o_resid=None, *, workspace=None, stream=None):
    """Forward on views: q, k, v share one row layout, o and o_resid another
    (both [B, N_o, H, N, D] views, written in place); lse [B, N_o, H, N] fp32
    contiguous.  Bitwise the same results as tri_attn_fwd on copies."""
    s = shape_of(q)
    B, No, H, N, D = q.shape
    lq, lo = layout_of(q), layout_of(o)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_view(t, name, (B, No, H, N, D), lq)
    for name, t in (("o", o), ("o_resid", o_resid)):
        if t is not None:
            _check_view(t, name, (B, No, H, N, D), lo)
    _check(bias, "bias", (B, H, N, N))
    _check(lse, "lse", (B, No, H, N), torch.float32)
    if mask is not None:
        _check(mask, "mask", (B, No, N))
    if workspace is None:
        need = fwd_workspace_bytes(s)
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device) if need > 0 else None
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = load().tri_attn_fwd_strided(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), ctypes.byref(lq), _ptr(bias),
                                       _ptr(mask), _ptr(o), _ptr(lse), _ptr(o_resid), ctypes.byref(lo),
                                       _ptr(workspace), ctypes.c_size_t(nbytes), _stream_ptr(stream))
    _raise(code, "tri_attn_fwd_strided")
    return o, lse, o_resid


def tri_attn_bwd_strided(q, k, v, bias, mask, o, o_resid, lse, do, dq, dk, dv, dbias, *, workspace=None,
                         stream=None):
    """Backward on views: q, k, v share one row layout, o and o_resid a
    second, do a third and dq, dk, dv a fourth; dq, dk, dv and dbias
    ([B, H, N, N] bf16) written in place."""
    s = shape_of(q)
    B, No, H, N, D = q.shape
    lq, lo, ldo, lg = layout_of(q), layout_of(o), layout_of(do), layout_of(dq)
    for name, t, lay in (("q", q, lq), ("k", k, lq), ("v", v, lq), ("dq", dq, lg), ("dk", dk, lg), ("dv", dv, lg),
                         ("o", o, lo), ("o_resid", o_resid, lo), ("do", do, ldo)):
        if t is not None:
            _check_view(t, name, (B, No, H, N, D), lay)
    _check(bias, "bias", (B, H, N, N))
    _check(dbias, "dbias", (B, H, N, N))
    _check(lse, "lse", (B, No, H, N), torch.float32)
    if mask is not None:
        _check(mask, "mask", (B, No, N))
    if workspace is None:
        workspace = torch.empty(bwd_workspace_bytes(s), dtype=torch.uint8, device=q.device)
    code = load().tri_attn_bwd_strided(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), ctypes.byref(lq), _ptr(bias),
                                       _ptr(mask), _ptr(o), _ptr(o_resid), ctypes.byref(lo), _ptr(lse), _ptr(do),
                                       ctypes.byref(ldo), _ptr(dq), _ptr(dk), _ptr(dv), ctypes.byref(lg),
                                       _ptr(dbias), _ptr(workspace),
                                       ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                       _stream_ptr(stream))
    _raise(code, "tri_attn_bwd_strided")
    return dq, dk, dv, dbias


ATOMIC_DQ, ATOMIC_DBIAS, ATOMIC_DBIAS_DQ, BULK_DQ, BULK_DQ_ATOMIC_DBIAS = 1, 2, 3, 4, 6


def bwd_atomic_workspace_bytes(q_or_shape, atomic_mask: int) -> int:
    """Workspace of the atomic ablation (0 for an invalid shape or mask)."""
    s = q_or_shape if isinstance(q_or_shape, Shape) else shape_of(q_or_shape)
    return int(load().triattn_bwd_atomic_workspace_bytes(ctypes.byref(s), int(atomic_mask)))


def tri_attn_bwd_atomic_ablation(q, k, v, bias, mask, o, o_resid, lse, do, atomic_mask=ATOMIC_DBIAS_DQ, *,
                                 workspace=None, out=None, stream=None):
    """Ablation only (not the library's backward): the backward with FP32
    atomics for dQ (``atomic_mask=1``), dbias (2) or both (3), or TMA bulk
    reductions for dQ (4; 6 with atomic dbias), instead of the ordered
    single-writer partials.  The gradients added that way are not bitwise
    reproducible between calls.  Returns (dq, dk, dv, dbias) in bf16."""
    s = shape_of(q)
    B, No, H, N, D = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check(t, name, (B, No, H, N, D))
    if o_resid is not None:
        _check(o_resid, "o_resid", (B, No, H, N, D))
    _check(bias, "bias", (B, H, N, N))
    _check(lse, "lse", (B, No, H, N), torch.float32)
    if mask is not None:
        _check(mask, "mask", (B, No, N))
    need = bwd_atomic_workspace_bytes(s, atomic_mask)
    if need == 0:
        raise TriAttnError(ERR_INVALID_ARG, "tri_attn_bwd_atomic_ablation")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        dbias = torch.empty_like(bias)
    else:
        dq, dk, dv, dbias = out
    code = load().tri_attn_bwd_atomic_ablation(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(mask),
                                               _ptr(o), _ptr(o_resid), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                                               _ptr(dv), _ptr(dbias), int(atomic_mask), _ptr(workspace),
                                               ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                               _stream_ptr(stream))
    _raise(code, "tri_attn_bwd_atomic_ablation")
    return dq, dk, dv, dbias


def tri_attn_dbias_combine(parts, *, out=None, stream=None):
    """dbias of an outer axis split across GPUs: ``parts`` is [R, B, H, N, N]
    FP32 (each written by tri_attn_bwd(..., dbias_fp32=True) on one shard,
    gathered in rank order); returns bf16 [B, H, N, N], the parts added in
    ascending r in FP32 and rounded once."""
    if parts.dim() != 5 or parts.dtype != torch.float32 or not parts.is_cuda or not parts.is_contiguous():
        raise ValueError("parts must be a contiguous CUDA float32 tensor [R, B, H, N, N]")
    R, B, H, N, N2 = parts.shape
    if N != N2:
        raise ValueError("parts must be [R, B, H, N, N]")
    s = Shape(B, N, N, H, 16, 0)
    dbias = out if out is not None else torch.empty((B, H, N, N), dtype=torch.bfloat16, device=parts.device)
    _check(dbias, "dbias", (B, H, N, N))
    code = load().tri_attn_dbias_combine(ctypes.byref(s), _ptr(parts), int(R), _ptr(dbias), _stream_ptr(stream))
    _raise(code, "tri_attn_dbias_combine")
    return dbias


def device_status(stream=None) -> int:
    """Synchronise the stream and return (then clear) the device status code."""
    return int(load().triattn_device_status(_stream_ptr(stream)))


def set_wait_limit_ns(ns: int) -> None:
    load().triattn_set_wait_limit_ns(ctypes.c_ulonglong(int(ns)))


def trace_enable(on: bool = True) -> None:
    """Start (clearing old records) or stop per-kernel CUDA-event tracing."""
    load().triattn_trace_enable(1 if on else 0)


def trace_read() -> dict:
    """Per-kernel totals of the traced launches: {name: {launches, total_ms,
    mean_ms, min_ms, max_ms}} (synchronises the recorded events)."""
    buf = (TraceEntry * 64)()
    n = load().triattn_trace_read(buf, 64)
    if n < 0:
        raise TriAttnError(ERR_CUDA, "triattn_trace_read")
    out = {}
    for e in buf[:n]:
        name = e.kernel.decode()
        out[name] = {"launches": e.launches, "total_ms": e.total_ms, "mean_ms": e.total_ms / max(e.launches, 1),
                     "min_ms": e.min_ms, "max_ms": e.max_ms}
    return out


def test_set_starve(on: bool) -> None:
    """Test hook: starve the forward's MMA warp so its bounded wait runs out."""
    load().triattn_test_set_starve(1 if on else 0)


def module_sizes(B: int, N: int, C: int, H: int, D: int):
    """(ctx bytes, workspace bytes) of the module; (0, 0) for an unsupported shape."""
    s = ModuleShape(B, N, C, H, D, 0)
    lib = load()
    return int(lib.triattn_module_ctx_bytes(ctypes.byref(s))), int(lib.triattn_module_workspace_bytes(ctypes.byref(s)))


def _module_shape(z, H, D):
    if z.dim() != 4 or z.shape[1] != z.shape[2]:
        raise ValueError("z must be [B, N, N, C]")
    B, N, _, C = z.shape
    return ModuleShape(B, N, C, H, D, 0)


def _bytes(t):
    return ctypes.c_size_t(t.numel() * t.element_size())


def tri_attn_module_fwd(z, mask, ln_w, ln_b, w_in, w_o, H: int, D: int, *, ctx=None, workspace=None, out=None,
                        stream=None):
    """Module forward: LayerNorm, projections into q, k, v and the bias, the
    core, output projection.  Returns (out [B, N, N, C] bf16, ctx) where ctx
    is the uint8 buffer the backward needs."""
    s = _module_shape(z, H, D)
    B, N, C = s.B, s.N, s.C
    F = 3 * H * D + H
    _check(z, "z", (B, N, N, C))
    _check(ln_w, "ln_w", (C,), torch.float32)
    _check(ln_b, "ln_b", (C,), torch.float32)
    _check(w_in, "w_in", (C, F))
    _check(w_o, "w_o", (H * D, C))
    if mask is not None:
        _check(mask, "mask", (B, N, N))
    nctx, nws = module_sizes(B, N, C, H, D)
    if nctx == 0:
        raise TriAttnError(ERR_UNSUPPORTED, "tri_attn_module_fwd")
    if ctx is None:
        ctx = torch.empty(nctx, dtype=torch.uint8, device=z.device)
    if workspace is None:
        workspace = torch.empty(nws, dtype=torch.uint8, device=z.device)
    if out is None:
        out = torch.empty_like(z)
    _check(out, "out", (B, N, N, C))
    code = load().tri_attn_module_fwd(ctypes.byref(s), _ptr(z), _ptr(mask), _ptr(ln_w), _ptr(ln_b), _ptr(w_in),
                                      _ptr(w_o), _ptr(out), _ptr(ctx), _ptr(workspace), _bytes(workspace),
                                      _stream_ptr(stream))
    _raise(code, "tri_attn_module_fwd")
    return out, ctx


def tri_attn_module_bwd(z, mask, ln_w, w_in, w_o, ctx, d_out, H: int, D: int, *, workspace=None, out=None,
                        stream=None):
    """Module backward of <out, d_out>.  Returns (dz bf16, d_ln_w, d_ln_b,
    d_w_in, d_w_o fp32)."""
    s = _module_shape(z, H, D)
    B, N, C = s.B, s.N, s.C
    F = 3 * H * D + H
    _check(z, "z", (B, N, N, C))
    _check(d_out, "d_out", (B, N, N, C))
    _check(ln_w, "ln_w", (C,), torch.float32)
    _check(w_in, "w_in", (C, F))
    _check(w_o, "w_o", (H * D, C))
    if mask is not None:
        _check(mask, "mask", (B, N, N))
    nctx, nws = module_sizes(B, N, C, H, D)
    if nctx == 0:
        raise TriAttnError(ERR_UNSUPPORTED, "tri_attn_module_bwd")
    _check(ctx, "ctx", (nctx,), torch.uint8)
    if workspace is None:
        workspace = torch.empty(nws, dtype=torch.uint8, device=z.device)
    if out is None:
        f32 = dict(dtype=torch.float32, device=z.device)
        out = (torch.empty_like(z), torch.empty(C, **f32), torch.empty(C, **f32), torch.empty((C, F), **f32),
               torch.empty((H * D, C), **f32))
    dz, dlw, dlb, dwi, dwo = out
    code = load().tri_attn_module_bwd(ctypes.byref(s), _ptr(z), _ptr(mask), _ptr(ln_w), _ptr(w_in), _ptr(w_o),
                                      _ptr(ctx), _ptr(d_out), _ptr(dz), _ptr(dlw), _ptr(dlb), _ptr(dwi), _ptr(dwo),
                                      _ptr(workspace), _bytes(workspace), _stream_ptr(stream))
    _raise(code, "tri_attn_module_bwd")
    return dz, dlw, dlb, dwi, dwo


def trimul_shape(B: int, N: int, Cz: int, Ch: int, direction: str) -> TriMulShape:
    if direction not in TRIMUL_DIRECTIONS:
        raise ValueError(f"direction must be one of {tuple(TRIMUL_DIRECTIONS)}")
    return TriMulShape(B, N, Cz, Ch, TRIMUL_DIRECTIONS[direction], 0)


def trimul_sizes(B: int, N: int, Cz: int, Ch: int, direction: str = "outgoing"):
    """(ctx bytes, workspace bytes) of the triangle multiplicative update; (0, 0)
    for an unsupported shape."""
    s = trimul_shape(B, N, Cz, Ch, direction)
    lib = load()
    return int(lib.triattn_trimul_ctx_bytes(ctypes.byref(s))), int(lib.triattn_trimul_workspace_bytes(ctypes.byref(s)))


def _trimul_check(z, mask, ln_in_w, w_p, ln_out_w, w_o):
    if z.dim() != 4 or z.shape[1] != z.shape[2]:
        raise ValueError("z must be [B, N, N, C_z]")
    B, N, _, Cz = z.shape
    if w_o.dim() != 2:
        raise ValueError("w_o must be [C_h, C_z]")
    Ch = w_o.shape[0]
    _check(z, "z", (B, N, N, Cz))
    _check(ln_in_w, "ln_in_w", (Cz,), torch.float32)
    _check(w_p, "w_p", (Cz, 4 * Ch + Cz))
    _check(ln_out_w, "ln_out_w", (Ch,), torch.float32)
    _check(w_o, "w_o", (Ch, Cz))
    if mask is not None:
        _check(mask, "mask", (B, N, N))
    return B, N, Cz, Ch


def triattn_trimul_fwd(z, mask, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o, direction: str, *, ctx=None,
                       workspace=None, out=None, stream=None):
    """Triangle multiplicative update forward ("outgoing" or "incoming").
    Returns (out [B, N, N, C_z] bf16, ctx) where ctx is the uint8 buffer the
    backward needs."""
    B, N, Cz, Ch = _trimul_check(z, mask, ln_in_w, w_p, ln_out_w, w_o)
    _check(ln_in_b, "ln_in_b", (Cz,), torch.float32)
    _check(ln_out_b, "ln_out_b", (Ch,), torch.float32)
    s = trimul_shape(B, N, Cz, Ch, direction)
    nctx, nws = trimul_sizes(B, N, Cz, Ch, direction)
    if nctx == 0:
        raise TriAttnError(ERR_UNSUPPORTED, "triattn_trimul_fwd")
    ctx = torch.empty(nctx, dtype=torch.uint8, device=z.device) if ctx is None else ctx
    workspace = torch.empty(nws, dtype=torch.uint8, device=z.device) if workspace is None else workspace
    out = torch.empty_like(z) if out is None else out
    _check(out, "out", (B, N, N, Cz))
    code = load().triattn_trimul_fwd(ctypes.byref(s), _ptr(z), _ptr(mask), _ptr(ln_in_w), _ptr(ln_in_b), _ptr(w_p),
                                     _ptr(ln_out_w), _ptr(ln_out_b), _ptr(w_o), _ptr(out), _ptr(ctx),
                                     _ptr(workspace), _bytes(workspace), _stream_ptr(stream))
    _raise(code, "triattn_trimul_fwd")
    return out, ctx


def triattn_trimul_bwd(z, mask, ln_in_w, w_p, ln_out_w, w_o, ctx, d_out, direction: str, *, workspace=None,
                       out=None, stream=None):
    """Backward of <out, d_out>.  Returns (dz bf16, d_ln_in_w, d_ln_in_b, d_w_p,
    d_ln_out_w, d_ln_out_b, d_w_o fp32)."""
    B, N, Cz, Ch = _trimul_check(z, mask, ln_in_w, w_p, ln_out_w, w_o)
    _check(d_out, "d_out", (B, N, N, Cz))
    s = trimul_shape(B, N, Cz, Ch, direction)
    nctx, nws = trimul_sizes(B, N, Cz, Ch, direction)
    if nctx == 0:
        raise TriAttnError(ERR_UNSUPPORTED, "triattn_trimul_bwd")
    _check(ctx, "ctx", (nctx,), torch.uint8)
    workspace = torch.empty(nws, dtype=torch.uint8, device=z.device) if workspace is None else workspace
    if out is None:
        f32 = dict(dtype=torch.float32, device=z.device)
        out = (torch.empty_like(z), torch.empty(Cz, **f32), torch.empty(Cz, **f32),
               torch.empty((Cz, 4 * Ch + Cz), **f32), torch.empty(Ch, **f32), torch.empty(Ch, **f32),
               torch.empty((Ch, Cz), **f32))
    dz, dliw, dlib, dwp, dlow, dlob, dwo = out
    code = load().triattn_trimul_bwd(ctypes.byref(s), _ptr(z), _ptr(mask), _ptr(ln_in_w), _ptr(w_p), _ptr(ln_out_w),
                                     _ptr(w_o), _ptr(ctx), _ptr(d_out), _ptr(dz), _ptr(dliw), _ptr(dlib), _ptr(dwp),
                                     _ptr(dlow), _ptr(dlob), _ptr(dwo), _ptr(workspace), _bytes(workspace),
                                     _stream_ptr(stream))
    _raise(code, "triattn_trimul_bwd")
    return out


def gemm(a, b, *, ta: bool = False, tb: bool = False, out_f32: bool = False, out=None, stream=None):
    """The library's tensor-core GEMM: op(a) @ op(b) for BF16 CUDA tensors,
    2-D or 3-D (batched, leading dimension), contiguous; op transposes the
    last two dimensions when ta / tb.  FP32 accumulation; BF16 output, or
    FP32 with ``out_f32``."""
    if a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16 or not (a.is_cuda and b.is_cuda):
        raise ValueError("a and b must be CUDA bfloat16 tensors")
    if a.dim() != b.dim() or a.dim() not in (2, 3) or not (a.is_contiguous() and b.is_contiguous()):
        raise ValueError("a and b must be contiguous, both 2-D or both 3-D")
    batched = a.dim() == 3
    a3, b3 = (a, b) if batched else (a[None], b[None])
    batch = a3.shape[0]
    M, K = (a3.shape[2], a3.shape[1]) if ta else (a3.shape[1], a3.shape[2])
    Kb, N = (b3.shape[2], b3.shape[1]) if tb else (b3.shape[1], b3.shape[2])
    if K != Kb or b3.shape[0] != batch:
        raise ValueError("shapes do not match")
    dt = torch.float32 if out_f32 else torch.bfloat16
    c = out if out is not None else torch.empty((batch, M, N), dtype=dt, device=a.device)
    lib = load()
    need = int(lib.triattn_gemm_workspace_bytes(M, N, K, batch))
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=a.device)
    code = lib.triattn_gemm(int(ta), int(tb), M, N, K, _ptr(a3), a3.shape[2], _ptr(b3), b3.shape[2], _ptr(c), N,
                            int(out_f32), batch, a3.shape[1] * a3.shape[2], b3.shape[1] * b3.shape[2], M * N,
                            _ptr(ws), ctypes.c_size_t(ws.numel()), _stream_ptr(stream))
    _raise(code, "triattn_gemm")
    return c if batched else c[0]


class TriAttnFunction(torch.autograd.Function):
    """Autograd wrapper: forward saves o, lse and the residual; backward runs
    the compensated key-tile-parallel backward."""

    @staticmethod
    def forward(ctx, q, k, v, bias, mask=None):
        o, lse, resid = tri_attn_fwd(q, k, v, bias, mask, save_residual=True)
        ctx.save_for_backward(q, k, v, bias, o, lse, resid)
        ctx.mask = mask
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, bias, o, lse, resid = ctx.saved_tensors
        dq, dk, dv, dbias = tri_attn_bwd(q, k, v, bias, ctx.mask, o, resid, lse, do.contiguous())
        return dq, dk, dv, dbias, None


def triangle_attention(q, k, v, bias, mask=None):
    """Differentiable triangular attention (BF16 in, BF16 out)."""
    return TriAttnFunction.apply(q, k, v, bias, mask)
