"""kkt_solve_fwd_noalloc, the entry point for callers that cannot allocate device memory.

Such callers (a framework that has handed all device memory to its own pool, an
operator that only receives its inputs and outputs, a serving loop that must not
synchronise on cudaMalloc) cannot supply the scratch workspace the tensor-core
kernel's work counter needs; this entry point keeps that counter in an array
compiled into the library instead.  Each test calls it through the C ABI twice in
a row on the same inputs and checks every result against the ordinary entry
point's output and against the fp64 oracle, under the tolerances of the other
parity tests.  After every call the counters in the array must be zero again.
One case has about 2000 tiles, far more than the GPU has SMs, so the counter
really hands out work and a counter left dirty by the first call would show in
the second.

This file is collected last on purpose, and passes alone in a fresh process or
after the whole suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gdn_chunkwise_ut_gb300 import _lib, device_status, kkt_solve_fwd
from gdn_chunkwise_ut_gb300.inputs import make_inputs
from tests.compare import check_T, check_WU, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _scratch_counters():
    out = (ctypes.c_ulonglong * 2)()
    assert _lib.lib().kkt_test_noalloc_scratch(ctypes.cast(out, ctypes.c_void_p)) == _lib.KKT_OK
    return list(out)


def _noalloc(k, v, beta, C, cu=None):
    Bt, T, H, dk = k.shape
    dv = v.shape[-1]
    T_out = torch.full((Bt, T, H, C), float("nan"), device=DEV)
    W = torch.full((Bt, T, H, dk), float("nan"), device=DEV, dtype=k.dtype)
    U = torch.full((Bt, T, H, dv), float("nan"), device=DEV, dtype=k.dtype)
    B = Bt if cu is None else cu.shape[0] - 1
    rc = _lib.lib().kkt_solve_fwd_noalloc(k.data_ptr(), v.data_ptr(), beta.data_ptr(),
                                          None if cu is None else cu.data_ptr(), B, T, H, dk, dv, C,
                                          T_out.data_ptr(), W.data_ptr(), U.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.KKT_OK, _lib.status_string(rc)
    torch.cuda.synchronize()
    assert device_status() == 0
    assert _scratch_counters() == [0, 0]
    return T_out, W, U


def _check(got, ref, oracle_out):
    """Within tolerance of the ordinary entry point's output and of the oracle's."""
    for g, r in ((got, ref), (got, oracle_out)):
        check_T(to64(g[0]), r[0] if isinstance(r[0], np.ndarray) else to64(r[0]))
        check_WU(to64(g[1]), r[1] if isinstance(r[1], np.ndarray) else to64(r[1]), "bf16", "W")
        check_WU(to64(g[2]), r[2] if isinstance(r[2], np.ndarray) else to64(r[2]), "bf16", "U")


def _oracle(k, v, beta, C, cu=None):
    return oracle.oracle_fwd(to64(k), to64(v), to64(beta), C,
                             cu_seqlens=None if cu is None else cu.cpu().numpy())


@pytest.mark.parametrize("C", [32, 64])
def test_noalloc_matches_default_entry_on_two_calls(C):
    k, v, beta = make_inputs(2, 1000, 4, 128, 128, seed=21 + C, device=DEV)  # ragged tail, 2 head groups
    ref = kkt_solve_fwd(k, v, beta, C)
    torch.cuda.synchronize()
    exact = _oracle(k, v, beta, C)
    for _ in range(2):
        _check(_noalloc(k, v, beta, C), ref, exact)


def test_noalloc_many_tiles_two_calls():
    """2 x 8192 tokens, 16 heads, C = 64: 2064 tiles, about 14 per SM, handed out by the counter."""
    k, v, beta = make_inputs(2, 8192, 16, 128, 128, seed=77, device=DEV)
    ref = kkt_solve_fwd(k, v, beta, 64)
    torch.cuda.synchronize()
    exact = _oracle(k, v, beta, 64)
    for _ in range(2):
        _check(_noalloc(k, v, beta, 64), ref, exact)


def test_noalloc_varlen_two_calls():
    lengths = [5, 64, 300, 1, 129]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=DEV)
    k, v, beta = make_inputs(1, int(sum(lengths)), 3, 128, 128, seed=31, device=DEV)
    ref = kkt_solve_fwd(k, v, beta, 64, cu)
    torch.cuda.synchronize()
    exact = _oracle(k, v, beta, 64, cu)
    for _ in range(2):
        _check(_noalloc(k, v, beta, 64, cu), ref, exact)


def test_noalloc_mixed_head_dims_and_unsupported_shapes():
    """d_k != d_v runs on the tensor-core kernel like any other covered shape; a head dimension
    outside {64, 128} is rejected."""
    lengths = [5, 64, 300, 1, 129]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=DEV)
    for dk, dv in ((64, 128), (128, 64)):
        k, v, beta = make_inputs(1, int(sum(lengths)), 3, dk, dv, seed=37, device=DEV)
        ref = kkt_solve_fwd(k, v, beta, 64, cu)
        torch.cuda.synchronize()
        exact = _oracle(k, v, beta, 64, cu)
        for _ in range(2):
            _check(_noalloc(k, v, beta, 64, cu), ref, exact)
    k = torch.zeros((1, 64, 1, 96), dtype=torch.bfloat16, device=DEV)
    v = torch.zeros((1, 64, 1, 128), dtype=torch.bfloat16, device=DEV)
    W, U = torch.zeros_like(k), torch.zeros_like(v)
    beta = torch.zeros((1, 64, 1), device=DEV)
    T_out = torch.zeros((1, 64, 1, 64), device=DEV)
    rc = _lib.lib().kkt_solve_fwd_noalloc(k.data_ptr(), v.data_ptr(), beta.data_ptr(), None, 1, 64, 1, 96, 128, 64,
                                          T_out.data_ptr(), W.data_ptr(), U.data_ptr(), None)
    assert rc == _lib.KKT_ERR_UNSUPPORTED
