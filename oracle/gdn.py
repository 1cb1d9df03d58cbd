"""ctypes front end of the fp64 C oracle of the GDN chunk state recurrence (``gdn_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU baseline.  The product path never imports it.

``recurrent_fwd`` is the token-by-token recurrence (the definition) and
``chunked_fwd`` the chunkwise form that consumes kkt_solve's W and U~; see the
header of ``gdn_oracle.c`` for the reading of the pages they follow.  This
module only marshals arrays: it converts its inputs to contiguous float64 and
hands them to C.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "gdn_oracle.c"
_LIB_PATH = _HERE / "_build" / "libgdn_oracle.so"
_lib = None

_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(src: Path | None = None, out: Path | None = None) -> Path:
    """Compile the oracle with gcc (OpenMP); ``src``/``out`` let mutation tests build a copy."""
    src = Path(src) if src is not None else _SRC
    out = Path(out) if out is not None else _LIB_PATH
    out.parent.mkdir(parents=True, exist_ok=True)
    if out == _LIB_PATH and out.exists() and out.stat().st_mtime >= src.stat().st_mtime:
        return out
    tmp = out.with_suffix(f".{os.getpid()}.tmp.so")
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", str(src), "-o", str(tmp), "-lm"],
                   check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    common = [ctypes.c_void_p, _i64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
              ctypes.c_int64]
    lib.gdn_oracle_recurrent.restype = ctypes.c_int
    lib.gdn_oracle_recurrent.argtypes = [_f64p, _f64p, _f64p, _f64p, ctypes.c_void_p] + common + \
        [ctypes.c_double, _f64p, ctypes.c_void_p, ctypes.c_int]
    lib.gdn_oracle_chunked.restype = ctypes.c_int
    lib.gdn_oracle_chunked.argtypes = [_f64p, _f64p, _f64p, _f64p, ctypes.c_void_p] + common + \
        [ctypes.c_int64, ctypes.c_double, _f64p, ctypes.c_void_p, ctypes.c_int]
    return lib


def load(path: Path | None = None):
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(str(path)))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(str(build())))
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _opt(a):
    return None if a is None else a.ctypes.data_as(_f64p)


def _layout(x, cu_seqlens, initial_state, H, dk, dv):
    Bt, T = x.shape[:2]
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        nseq, Ttot, cu_p = cu.shape[0] - 1, Bt * T, cu.ctypes.data_as(_i64p)
    else:
        cu, nseq, Ttot, cu_p = None, Bt, T, None
    h0 = None if initial_state is None else _f64(initial_state).reshape(nseq, H, dk, dv)
    return cu, nseq, Ttot, cu_p, h0


def recurrent_fwd(q, k, v, beta, g=None, initial_state=None, scale=1.0, cu_seqlens=None, nthreads=0, lib=None):
    """q, k [B, T, H, dk], v [B, T, H, dv], beta (and g) [B, T, H]; with ``cu_seqlens`` the tensors
    are [1, T, H, .].  ``initial_state`` [nseq, H, dk, dv] or None (zero).
    Returns (o [B, T, H, dv], final_state [nseq, H, dk, dv]) in float64."""
    lib = lib or load()
    q, k, v, beta = _f64(q), _f64(k), _f64(v), _f64(beta)
    g = None if g is None else _f64(g)
    H, dk, dv = k.shape[2], k.shape[3], v.shape[3]
    cu, nseq, Ttot, cu_p, h0 = _layout(k, cu_seqlens, initial_state, H, dk, dv)
    o = np.zeros(v.shape)
    ht = np.zeros((nseq, H, dk, dv))
    rc = lib.gdn_oracle_recurrent(q.ctypes.data_as(_f64p), k.ctypes.data_as(_f64p), v.ctypes.data_as(_f64p),
                                  beta.ctypes.data_as(_f64p), _opt(g), _opt(h0), cu_p, nseq, Ttot, H, dk, dv,
                                  float(scale), o.ctypes.data_as(_f64p), ht.ctypes.data_as(_f64p), int(nthreads))
    if rc != 0:
        raise ValueError(f"gdn_oracle_recurrent failed ({rc})")
    return o, ht


def chunked_fwd(q, k, w, u, C: int, g=None, initial_state=None, scale=1.0, cu_seqlens=None, nthreads=0, lib=None):
    """The chunkwise form from kkt_solve's W [B, T, H, dk] and U~ [B, T, H, dv] (same layouts as
    ``recurrent_fwd``).  Returns (o, final_state) in float64."""
    lib = lib or load()
    q, k, w, u = _f64(q), _f64(k), _f64(w), _f64(u)
    g = None if g is None else _f64(g)
    H, dk, dv = k.shape[2], k.shape[3], u.shape[3]
    cu, nseq, Ttot, cu_p, h0 = _layout(k, cu_seqlens, initial_state, H, dk, dv)
    o = np.zeros(u.shape)
    ht = np.zeros((nseq, H, dk, dv))
    rc = lib.gdn_oracle_chunked(q.ctypes.data_as(_f64p), k.ctypes.data_as(_f64p), w.ctypes.data_as(_f64p),
                                u.ctypes.data_as(_f64p), _opt(g), _opt(h0), cu_p, nseq, Ttot, H, dk, dv, int(C),
                                float(scale), o.ctypes.data_as(_f64p), ht.ctypes.data_as(_f64p), int(nthreads))
    if rc != 0:
        raise ValueError(f"gdn_oracle_chunked failed ({rc})")
    return o, ht
