"""kkt_solve_fwd_host's host-side logic (no GPU): the workspace size and the argument checks, which
return their status before any CUDA call."""
import ctypes

import numpy as np

from gdn_chunkwise_ut_gb300 import _lib


def _ws(B, T, H, dk, dv, C, io=0, gated=0, varlen=0, pieces=8):
    return _lib.lib().kkt_host_workspace_bytes(B, T, H, dk, dv, C, io, gated, varlen, pieces)


def _align(x):
    return (x + 255) // 256 * 256


def test_workspace_bytes_cover_every_tensor():
    B, T, H, dk, dv, C, P = 4, 8192, 16, 128, 128, 64, 8
    rows = B * T * H
    expect = (_align(256) + _align(rows * 2 * dk) + _align(rows * 2 * dv) + _align(rows * 4) + 0
              + _align(rows * 4 * C) + _align(rows * 2 * dk) + _align(rows * 2 * dv) + _align(4 * (B + 2 * P)))
    assert _ws(B, T, H, dk, dv, C, pieces=P) == expect
    # gated adds g, fp16 T halves T, fp32 I/O doubles k, v, W, U, varlen counts T rows
    assert _ws(B, T, H, dk, dv, C, gated=1, pieces=P) == expect + _align(rows * 4)
    assert _ws(B, T, H, dk, dv, C, io=0x100, pieces=P) == expect - _align(rows * 4 * C) + _align(rows * 2 * C)
    assert _ws(B, T, H, dk, dv, C, io=1, pieces=P) > expect
    assert _ws(32, 156617, 32, 128, 128, 64, varlen=1) < _ws(1, 156617 * 32, 32, 128, 128, 64)


def test_workspace_bytes_reject_bad_sizes():
    assert _ws(0, 10, 1, 64, 64, 64) == 0
    assert _ws(1, 10, 1, 64, 64, 64, pieces=0) == 0
    assert _ws(1, 10, 1, 64, 64, 64, pieces=_lib.KKT_HOST_MAX_PIECES + 1) == 0


def _call(cu=None, B=2, T=100, ws_bytes=1 << 40, ws=256, pieces=4, C=64, dk=128):
    # host pointers that are never dereferenced: every check below fails before any copy
    dummy = ctypes.c_void_p(4096)
    cu_ptr = None if cu is None else cu.ctypes.data_as(ctypes.c_void_p)
    return _lib.lib().kkt_solve_fwd_host(dummy, dummy, dummy, None, cu_ptr, B, T, 3, dk, 128, C, dummy, dummy,
                                         dummy, 0, 0, pieces, ctypes.c_void_p(ws), ws_bytes, None)


def test_argument_errors_before_any_cuda_call():
    assert _call(ws_bytes=1024) == _lib.KKT_ERR_ARG            # workspace too small
    assert _call(ws=4096 + 16) == _lib.KKT_ERR_ARG             # workspace not 256-byte aligned
    assert _call(pieces=0) == _lib.KKT_ERR_ARG
    assert _call(pieces=_lib.KKT_HOST_MAX_PIECES + 1) == _lib.KKT_ERR_ARG
    assert _call(C=48) == _lib.KKT_ERR_UNSUPPORTED
    assert _call(dk=96) == _lib.KKT_ERR_UNSUPPORTED
    bad = np.array([0, 50, 40, 100], dtype=np.int32)           # decreasing
    assert _call(cu=bad, B=3, T=100) == _lib.KKT_ERR_SEQLENS
    short = np.array([0, 50, 90], dtype=np.int32)              # does not end at T
    assert _call(cu=short, B=2, T=100) == _lib.KKT_ERR_SEQLENS
