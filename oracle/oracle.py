"""Python front end of the FP64 CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product package never does.

The arithmetic lives in ``triattn_oracle.c`` (plain C, OpenMP over slices);
this file only compiles it with gcc, loads it with ctypes and converts
arrays to contiguous float64.  See ``triattn_oracle.c`` for the definition
and its sources in "TurboPairFormer: Fast and Stable Protein Folding Model
Training with an Optimized Triangle Attention Kernel" (Abstract, Figure 1(a),
Table 1, Figure 6).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "triattn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = None
_LOCK = threading.Lock()


class _Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("No", ctypes.c_int), ("H", ctypes.c_int),
                ("Nq", ctypes.c_int), ("Nk", ctypes.c_int), ("D", ctypes.c_int)]


def lib_path() -> str:
    return os.path.join(_BUILD, f"libtriattn_oracle_{platform.machine()}.so")


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc -O2 -fopenmp) if stale."""
    out = lib_path()
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    sp = ctypes.POINTER(_Shape)
    lib.oracle_fwd.argtypes = [sp, dp, dp, dp, dp, dp, dp, dp]
    lib.oracle_fwd.restype = None
    lib.oracle_bwd.argtypes = [sp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp]
    lib.oracle_bwd.restype = None
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            _LIB = _declare(ctypes.CDLL(build()))
    return _LIB


def compile_variant(source_text: str, tag: str) -> str:
    """Compile an edited copy of the oracle source (used by tests that plant
    a mistake in the oracle to show the pins catch it).  Returns the path."""
    # a private temporary folder, so that planted variants never pile up
    # next to the oracle's own build
    d = tempfile.mkdtemp(prefix=f"oracle_variant_{tag}_")
    src = os.path.join(d, "variant.c")
    out = os.path.join(d, f"libvariant_{platform.machine()}.so")
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c99", src, "-o", out, "-lm"], check=True)
    return out


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _f64(x) -> np.ndarray:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape(q, k):
    B, No, H, Nq, D = q.shape
    Bk, Nok, Hk, Nk, Dk = k.shape
    assert (B, No, H, D) == (Bk, Nok, Hk, Dk), "q/k shapes disagree"
    return _Shape(B, No, H, Nq, Nk, D)


def load_variant(path: str):
    """Load a compiled oracle variant; pass the result as ``lib=``."""
    return _declare(ctypes.CDLL(path))


def max_threads() -> int:
    return int(_lib().oracle_max_threads())


def fwd(q, k, v, bias, mask=None, lib=None):
    """Exact forward.  Returns (O [B,No,H,Nq,D], lse [B,No,H,Nq]) in float64."""
    q, k, v, bias, mask = map(_f64, (q, k, v, bias, mask))
    s = _shape(q, k)
    assert bias.shape == (s.B, s.H, s.Nq, s.Nk)
    if mask is not None:
        assert mask.shape == (s.B, s.No, s.Nk)
    o = np.empty(q.shape, np.float64)
    lse = np.empty(q.shape[:-1], np.float64)
    (lib or _lib()).oracle_fwd(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(mask), _ptr(o), _ptr(lse))
    return o, lse


def bwd(q, k, v, bias, mask, dO, lib=None):
    """Exact gradients of sum(dO * O).  Returns (dq, dk, dv, dbias) in float64."""
    q, k, v, bias, mask, dO = map(_f64, (q, k, v, bias, mask, dO))
    s = _shape(q, k)
    assert bias.shape == (s.B, s.H, s.Nq, s.Nk) and dO.shape == q.shape
    if mask is not None:
        assert mask.shape == (s.B, s.No, s.Nk)
    dq = np.empty(q.shape, np.float64)
    dk = np.empty(k.shape, np.float64)
    dv = np.empty(v.shape, np.float64)
    dbias = np.empty(bias.shape, np.float64)
    (lib or _lib()).oracle_bwd(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(mask), _ptr(dO),
                      _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias))
    return dq, dk, dv, dbias


def rows(q, k, v, bias, mask, dO, b, h, qrows):
    """Exact O, lse, dQ and dbias restricted to query rows ``qrows`` of head
    ``(b, h)``, over every slice o.  Uses the Nq != Nk generality of the
    oracle: only the selected rows of Q, bias and dO enter.

    Returns dict with o [No,R,D], lse [No,R], dq [No,R,D], dbias [R,Nk].
    """
    qrows = np.asarray(qrows, dtype=np.int64)
    q, k, v, bias, mask, dO = map(_f64, (q, k, v, bias, mask, dO))
    qs = np.ascontiguousarray(q[b:b + 1, :, h:h + 1][:, :, :, qrows])
    ks = np.ascontiguousarray(k[b:b + 1, :, h:h + 1])
    vs = np.ascontiguousarray(v[b:b + 1, :, h:h + 1])
    gs = np.ascontiguousarray(dO[b:b + 1, :, h:h + 1][:, :, :, qrows])
    bs = np.ascontiguousarray(bias[b:b + 1, h:h + 1][:, :, qrows])
    ms = None if mask is None else np.ascontiguousarray(mask[b:b + 1])
    o, lse = fwd(qs, ks, vs, bs, ms)
    dq, _, _, db = bwd(qs, ks, vs, bs, ms, gs)
    return {"o": o[0, :, 0], "lse": lse[0, :, 0], "dq": dq[0, :, 0], "dbias": db[0, 0]}


def slice_(q, k, v, bias, mask, dO, b, o, h):
    """Exact results of one slice (b, o, h): O, lse, dQ, dK, dV and that
    slice's own dS (its contribution to dbias)."""
    q, k, v, bias, mask, dO = map(_f64, (q, k, v, bias, mask, dO))
    sl = (slice(b, b + 1), slice(o, o + 1), slice(h, h + 1))
    qs, ks, vs, gs = (np.ascontiguousarray(t[sl]) for t in (q, k, v, dO))
    bs = np.ascontiguousarray(bias[b:b + 1, h:h + 1])
    ms = None if mask is None else np.ascontiguousarray(mask[b:b + 1, o:o + 1])
    out, lse = fwd(qs, ks, vs, bs, ms)
    dq, dk, dv, ds = bwd(qs, ks, vs, bs, ms, gs)
    return {"o": out[0, 0, 0], "lse": lse[0, 0, 0], "dq": dq[0, 0, 0], "dk": dk[0, 0, 0],
            "dv": dv[0, 0, 0], "ds": ds[0, 0]}
