"""kkt_solve_fwd_noalloc, the entry point for callers that cannot allocate device memory.

Such callers (a framework that has handed all device memory to its own pool, an
operator that only receives its inputs and outputs, a serving loop that must not
synchronise on cudaMalloc) cannot supply the scratch workspace the tensor-core
kernel's work counter needs; this entry point keeps that counter in an array
compiled into the library instead.  The test calls it through the C ABI, twice in
a row on the same inputs (the second call must see its counter cleared, not the
value the first call left), and compares each result with the ordinary entry
point's output under the same tolerances as the other parity tests.

This file is collected last on purpose, and passes alone in a fresh process or
after the whole suite.
"""
import numpy as np
import pytest
import torch

from gdn_chunkwise_ut_gb300 import _lib, device_status, kkt_solve_fwd
from gdn_chunkwise_ut_gb300.inputs import make_inputs
from tests.compare import check_T, check_WU, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


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
    return T_out, W, U


def _same_within_tolerance(got, ref):
    check_T(to64(got[0]), to64(ref[0]))
    check_WU(to64(got[1]), to64(ref[1]), "bf16", "W")
    check_WU(to64(got[2]), to64(ref[2]), "bf16", "U")


@pytest.mark.parametrize("C", [32, 64])
def test_noalloc_matches_default_entry_on_two_calls(C):
    k, v, beta = make_inputs(2, 1000, 4, 128, 128, seed=21 + C, device=DEV)  # ragged tail, 2 head groups
    ref = kkt_solve_fwd(k, v, beta, C)
    torch.cuda.synchronize()
    for _ in range(2):
        _same_within_tolerance(_noalloc(k, v, beta, C), ref)


def test_noalloc_varlen_two_calls():
    lengths = [5, 64, 300, 1, 129]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=DEV)
    k, v, beta = make_inputs(1, int(sum(lengths)), 3, 128, 128, seed=31, device=DEV)
    ref = kkt_solve_fwd(k, v, beta, 64, cu)
    torch.cuda.synchronize()
    for _ in range(2):
        _same_within_tolerance(_noalloc(k, v, beta, 64, cu), ref)


def test_noalloc_mixed_head_dims_and_unsupported_shapes():
    """d_k != d_v runs on the tensor-core kernel like any other covered shape; a head dimension
    outside {64, 128} is rejected."""
    lengths = [5, 64, 300, 1, 129]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=DEV)
    for dk, dv in ((64, 128), (128, 64)):
        k, v, beta = make_inputs(1, int(sum(lengths)), 3, dk, dv, seed=37, device=DEV)
        ref = kkt_solve_fwd(k, v, beta, 64, cu)
        torch.cuda.synchronize()
        _same_within_tolerance(_noalloc(k, v, beta, 64, cu), ref)
    k = torch.zeros((1, 64, 1, 96), dtype=torch.bfloat16, device=DEV)
    v = torch.zeros((1, 64, 1, 128), dtype=torch.bfloat16, device=DEV)
    W, U = torch.zeros_like(k), torch.zeros_like(v)
    beta = torch.zeros((1, 64, 1), device=DEV)
    T_out = torch.zeros((1, 64, 1, 64), device=DEV)
    rc = _lib.lib().kkt_solve_fwd_noalloc(k.data_ptr(), v.data_ptr(), beta.data_ptr(), None, 1, 64, 1, 96, 128, 64,
                                          T_out.data_ptr(), W.data_ptr(), U.data_ptr(), None)
    assert rc == _lib.KKT_ERR_UNSUPPORTED
