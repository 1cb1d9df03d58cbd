"""ctypes declarations of libkkt.so (the C ABI in include/kkt.h).

Argument marshalling only.  If the library is missing, every entry point
raises: there is no Python or CPU fallback.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "_build" / "libkkt.so"

KKT_OK = 0
KKT_ERR_ARG = 1
KKT_ERR_UNSUPPORTED = 2
KKT_ERR_ALIGN = 3
KKT_ERR_CUDA = 4
KKT_ERR_SEQLENS = 5
KKT_ERR_TIMEOUT = 6
KKT_ERR_NO_DEVICE = 7

KKT_IO_BF16 = 0
KKT_IO_F32 = 1
KKT_T_OUT_F16 = 0x100  # ORed into the io dtype: T_out in fp16

KKT_KERNEL_AUTO = 0
KKT_KERNEL_SIMT = 1
KKT_KERNEL_TC = 2

KERNELS = {"auto": KKT_KERNEL_AUTO, "simt": KKT_KERNEL_SIMT, "tc": KKT_KERNEL_TC}

KKT_WORKSPACE_BYTES = 256
KKT_HOST_MAX_PIECES = 64
KKT_NOALLOC_SCRATCH_BYTES = 256

_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t

SIGNATURES = {
    "kkt_solve_fwd": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "kkt_solve_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _i, _i, _vp, _sz, _vp]),
    "kkt_solve_fwd_gated": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _i, _i, _vp, _sz,
                                 _vp]),
    "kkt_solve_fwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "gdn_chunk_state_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, ctypes.c_float, _vp,
                                 _vp, _vp]),
    "kkt_host_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i, _i, _i]),
    "kkt_solve_fwd_host": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _i, _i, _i, _vp, _sz,
                                _vp]),
    "kkt_test_stalled_solve": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "kkt_test_noalloc_scratch": (_i, [_vp]),
    "kkt_test_plan_pieces": (_i, [_vp, _i, _i, _i, _vp, _vp, _i, _vp, _i]),
    "kkt_device_status": (_i, [_vp]),
    "kkt_debug_bounds": (_i, [_vp, _vp]),
    "kkt_select_kernel": (_i, [_i, _i, _i, _i, _i]),
    "kkt_status_string": (ctypes.c_char_p, [_i]),
    "kkt_version": (_i, []),
}


class KktError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = status_string(status) if LIB_PATH.exists() else f"status {status}"
        super().__init__(f"{what}: {msg} (kkt_status {status})" if what else f"{msg} (kkt_status {status})")


_lib = None


def lib(path: Path | None = None):
    """The loaded library (raises if it has not been built)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(str(path)))
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"libkkt.so is not built ({LIB_PATH}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        _lib = _declare(ctypes.CDLL(str(LIB_PATH)))
    return _lib


def _declare(l):
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(l, name)
        fn.restype = res
        fn.argtypes = args
    return l


def status_string(status: int) -> str:
    return lib().kkt_status_string(int(status)).decode()
