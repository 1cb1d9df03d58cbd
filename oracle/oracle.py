"""ctypes front end of the fp64 C oracle (``kkt_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU baseline.  The product path never imports it.

The oracle follows "TileLang 实战：单位下三角矩阵求逆" §1 (A, W, U~), §2.1 (row
forward substitution), §3.2 (beta on rows, unit diagonal) and §5 item 12 (the
gated coefficient); see the header of ``kkt_oracle.c``.  This module only marshals arrays: it converts its inputs to
contiguous float64 and hands them to C.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "kkt_oracle.c"
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "liboracle.so"
_lib = None

_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(src: Path | None = None, out: Path | None = None, extra_flags=()) -> Path:
    """Compile the oracle with gcc (OpenMP) into a shared library; returns its path.

    ``src``/``out`` let the mutation tests compile a modified copy elsewhere.
    """
    src = Path(src) if src is not None else _SRC
    out = Path(out) if out is not None else _LIB_PATH
    out.parent.mkdir(parents=True, exist_ok=True)
    if out == _LIB_PATH and out.exists() and out.stat().st_mtime >= src.stat().st_mtime:
        return out
    tmp = out.with_suffix(f".{os.getpid()}.tmp.so")
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           *extra_flags, str(src), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    lib.kkt_oracle_chunk.restype = ctypes.c_int
    lib.kkt_oracle_chunk.argtypes = [_f64p, _f64p, _f64p, _f64p, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, _f64p, _f64p, _f64p, _f64p]
    lib.kkt_oracle_fwd.restype = ctypes.c_int
    lib.kkt_oracle_fwd.argtypes = [_f64p, _f64p, _f64p, _f64p, _i64p] + [ctypes.c_int64] * 6 + \
        [_f64p, _f64p, _f64p, ctypes.c_int]
    lib.kkt_oracle_threads.restype = ctypes.c_int
    lib.kkt_oracle_threads.argtypes = [ctypes.c_int]
    return lib


def load(path: Path | None = None):
    """Load (building if needed) the oracle library.  ``path`` loads another build."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(str(path)))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(str(build())))
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_f64p)


def oracle_chunk(k, v, beta, C: int, lib=None, g=None):
    """One chunk of Lc <= C rows.

    k [Lc, dk], v [Lc, dv], beta [Lc] -> (T [Lc, C], W [Lc, dk], U [Lc, dv], A [C, C]).
    ``g`` [Lc]: per-token log decays of the gated variant (None: ungated).
    """
    lib = lib or load()
    k, v, beta = _f64(k), _f64(v), _f64(beta)
    g = None if g is None else _f64(g)
    Lc, dk = k.shape
    dv = v.shape[1]
    T = np.empty((Lc, C)); W = np.empty((Lc, dk)); U = np.empty((Lc, dv)); A = np.empty((C, C))
    rc = lib.kkt_oracle_chunk(_ptr(k), _ptr(v), _ptr(beta), None if g is None else _ptr(g), Lc, C, dk, dv,
                              _ptr(T), _ptr(W), _ptr(U), _ptr(A))
    if rc != 0:
        raise ValueError(f"kkt_oracle_chunk failed ({rc})")
    return T, W, U, A


def oracle_fwd(k, v, beta, C: int, cu_seqlens=None, nthreads: int = 0, lib=None, g=None):
    """Whole tensors in the library's layout.

    k [B, T, H, dk], v [B, T, H, dv], beta [B, T, H]; with ``cu_seqlens`` (B+1
    offsets) the tensors are [1, T, H, .] and hold B packed sequences.  ``g``
    [B, T, H]: per-token log decays of the gated variant (None: ungated).
    Returns (T_out [B, T, H, C], W [B, T, H, dk], U [B, T, H, dv]) in float64.
    """
    lib = lib or load()
    k, v, beta = _f64(k), _f64(v), _f64(beta)
    g = None if g is None else _f64(g)
    Bt, T, H, dk = k.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        B = cu.shape[0] - 1
        cu_p = cu.ctypes.data_as(_i64p)
        Ttot = Bt * T
    else:
        B, Ttot, cu_p, cu = Bt, T, None, None
    T_out = np.zeros((Bt, T, H, C)); W = np.zeros((Bt, T, H, dk)); U = np.zeros((Bt, T, H, dv))
    rc = lib.kkt_oracle_fwd(_ptr(k), _ptr(v), _ptr(beta), None if g is None else _ptr(g), cu_p,
                            B, Ttot, H, dk, dv, C,
                            _ptr(T_out), _ptr(W), _ptr(U), int(nthreads))
    if rc != 0:
        raise ValueError(f"kkt_oracle_fwd failed ({rc})")
    return T_out, W, U


def oracle_threads(nthreads: int = 0, lib=None) -> int:
    lib = lib or load()
    return int(lib.kkt_oracle_threads(int(nthreads)))


if __name__ == "__main__":  # pragma: no cover
    print(build())
    sys.exit(0)
