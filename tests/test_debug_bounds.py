"""The bounds-checked build on the GPU (compute-sanitizer is not available where this runs).

libkkt_bounds.so is the library built with -DKKT_DEBUG_BOUNDS (kkt_debug.cuh): every shared-memory
access of the tensor-core kernel, every array access of the SIMT kernel and every plain global load
and store of both are checked against their ranges, and a failed check is counted and redirected
(no fault, no trap).  These tests run that build over the shapes that exercise the edges (short
last chunks, empty and one-token sequences, a partial head group, every chunk size, both kernels,
the gated, fp16-T and W/U-only variants), check that no access left its range, and compare the
results with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from gdn_chunkwise_ut_gb300 import _lib, build
from gdn_chunkwise_ut_gb300.inputs import make_gate, make_inputs
from tests.compare import check_T, check_WU, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def blib():
    lib = _lib.lib(build.build(debug_bounds=True))
    assert lib.kkt_debug_bounds(None, None) >= 0  # a bounds-checked build; clears the records
    return lib


def _call(lib, k, v, beta, C, cu, kernel, g=None, t_dtype=torch.float32, with_t=True):
    Bt, T, H, dk = k.shape
    dv = v.shape[-1]
    T_out = torch.full((Bt, T, H, C), float("nan"), device=DEV, dtype=t_dtype) if with_t else None
    W = torch.full((Bt, T, H, dk), float("nan"), device=DEV, dtype=k.dtype)
    U = torch.full((Bt, T, H, dv), float("nan"), device=DEV, dtype=k.dtype)
    cu_t = None if cu is None else torch.as_tensor(np.asarray(cu), dtype=torch.int32, device=DEV)
    B = Bt if cu is None else len(cu) - 1
    io = (_lib.KKT_IO_F32 if k.dtype == torch.float32 else _lib.KKT_IO_BF16) | \
        (_lib.KKT_T_OUT_F16 if t_dtype == torch.float16 else 0)
    ws = torch.zeros(_lib.KKT_WORKSPACE_BYTES // 4, dtype=torch.int32, device=DEV)
    rc = lib.kkt_solve_fwd_gated(k.data_ptr(), v.data_ptr(), beta.data_ptr(), None if g is None else g.data_ptr(),
                                 None if cu_t is None else cu_t.data_ptr(), B, T, H, dk, dv, C,
                                 None if T_out is None else T_out.data_ptr(), W.data_ptr(), U.data_ptr(), io,
                                 _lib.KERNELS[kernel], ws.data_ptr(), ws.numel() * 4,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.KKT_OK
    torch.cuda.synchronize()
    assert lib.kkt_device_status(None) == 0
    return T_out, W, U


def _no_violations(lib):
    first = np.zeros(1, dtype=np.uint64)
    kind = np.zeros(1, dtype=np.int32)
    n = lib.kkt_debug_bounds(first.ctypes.data, kind.ctypes.data)
    assert n == 0, f"{n} out-of-range accesses, first kind {int(kind[0])} at {int(first[0])}"


@pytest.mark.parametrize("kernel", ["tc", "simt"])
@pytest.mark.parametrize("C", [32, 64, 128])
@pytest.mark.parametrize("variant", ["plain", "gated", "t_fp16", "no_t"])
def test_in_range_and_correct(blib, kernel, C, variant):
    lengths = [1, 63, 64, 65, 0, 130, 7, 200, 128]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    k, v, beta = make_inputs(1, int(cu[-1]), 3, 128, 128, seed=C + 61, device=DEV)
    g = make_gate(1, int(cu[-1]), 3, seed=C + 61, device=DEV) if variant == "gated" else None
    t_dtype = torch.float16 if variant == "t_fp16" else torch.float32
    T_out, W, U = _call(blib, k, v, beta, C, cu, kernel, g=g, t_dtype=t_dtype, with_t=variant != "no_t")
    _no_violations(blib)
    T_ref, W_ref, U_ref = oracle.oracle_fwd(to64(k), to64(v), to64(beta), C, cu_seqlens=cu,
                                            g=None if g is None else to64(g))
    if T_out is not None:
        T_g = to64(T_out)
        if t_dtype == torch.float16:
            assert (np.abs(T_g - T_ref) <= 1e-4 + 2.0 ** -11 * np.abs(T_ref)).all()
        else:
            check_T(T_g, T_ref)
    check_WU(to64(W), W_ref, "bf16", "W")
    check_WU(to64(U), U_ref, "bf16", "U")


@pytest.mark.parametrize("C", [32, 64, 128])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (64, 128)])
def test_tc_head_dims(blib, C, dk, dv):
    lengths = [1, 63, 64, 65, 0, 130, 7, 200, 128]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    k, v, beta = make_inputs(1, int(cu[-1]), 3, dk, dv, seed=C + 95, device=DEV)
    g = make_gate(1, int(cu[-1]), 3, seed=C + 95, device=DEV)
    T_out, W, U = _call(blib, k, v, beta, C, cu, "tc", g=g)
    _no_violations(blib)
    T_ref, W_ref, U_ref = oracle.oracle_fwd(to64(k), to64(v), to64(beta), C, cu_seqlens=cu, g=to64(g))
    check_T(to64(T_out), T_ref)
    check_WU(to64(W), W_ref, "bf16", "W")
    check_WU(to64(U), U_ref, "bf16", "U")


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_fixed_length_partial_head_group(blib, kernel):
    """Fixed-length batch with a ragged tail and an odd head count (the last head group of the
    tensor-core kernel's tiles runs past H)."""
    k, v, beta = make_inputs(2, 3 * 64 + 17, 5, 128, 128, seed=71, device=DEV)
    T_out, W, U = _call(blib, k, v, beta, 64, None, kernel)
    _no_violations(blib)
    T_ref, W_ref, U_ref = oracle.oracle_fwd(to64(k), to64(v), to64(beta), 64)
    check_T(to64(T_out), T_ref)
    check_WU(to64(W), W_ref, "bf16", "W")
    check_WU(to64(U), U_ref, "bf16", "U")


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
def test_simt_head_dims_and_fp32(blib, dk, dv):
    k, v, beta = make_inputs(1, 150, 2, dk, dv, seed=72, device=DEV)
    T_out, W, U = _call(blib, k, v, beta, 64, None, "simt")
    _no_violations(blib)
    T_ref, W_ref, U_ref = oracle.oracle_fwd(to64(k), to64(v), to64(beta), 64)
    check_T(to64(T_out), T_ref)
    check_WU(to64(W), W_ref, "bf16", "W")
    kf, vf, bf = make_inputs(1, 128, 1, 64, 64, seed=73, dtype=torch.float32, device=DEV)
    T_out, W, U = _call(blib, kf, vf, bf, 32, None, "simt")
    _no_violations(blib)
    T_ref, W_ref, U_ref = oracle.oracle_fwd(to64(kf), to64(vf), to64(bf), 32)
    check_T(to64(T_out), T_ref)
    check_WU(to64(W), W_ref, "f32", "W")
