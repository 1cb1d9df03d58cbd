"""Failure detection of the tensor-core kernel on the GPU, without a GPU fault (GPU).

kkt_test_stalled_solve launches the kernel with the shared-memory stage of each CTA's
first tile never filled.  Every wait in the kernel is bounded, so the roles waiting on
that stage give up after their limit, record KKT_ERR_TIMEOUT, stop the rest of their CTA
and return; nothing faults, traps or waits without a bound.  The test checks the status
the host reads back, that the kernel ended within a few seconds, and that the context is
still usable: a normal call right after it matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from gdn_chunkwise_ut_gb300 import _lib, device_status, kkt_solve_fwd
from gdn_chunkwise_ut_gb300.inputs import make_inputs
from tests.compare import check_T, check_WU, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("C", [64, 128])
def test_stalled_stage_times_out_and_context_survives(C):
    k, v, beta = make_inputs(2, 300, 3, 128, 128, seed=13, device=DEV)
    T_out = torch.zeros((2, 300, 3, C), device=DEV)
    W = torch.zeros_like(k)
    U = torch.zeros_like(v)
    torch.cuda.synchronize()
    assert device_status() == _lib.KKT_OK  # also clears anything an earlier test left
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.monotonic()
    rc = _lib.lib().kkt_test_stalled_solve(k.data_ptr(), v.data_ptr(), beta.data_ptr(), None, 2, 300, 3, 128, 128,
                                           C, T_out.data_ptr(), W.data_ptr(), U.data_ptr(), stream)
    assert rc == _lib.KKT_OK
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert device_status() == _lib.KKT_ERR_TIMEOUT
    assert elapsed < 30.0, elapsed  # bounded waits of 2 s each, not a hang
    # the status word was read and cleared, and the context still computes correctly
    assert device_status() == _lib.KKT_OK
    T_g, W_g, U_g = kkt_solve_fwd(k, v, beta, C)
    torch.cuda.synchronize()
    assert device_status() == _lib.KKT_OK
    T_ref, W_ref, U_ref = oracle.oracle_fwd(to64(k), to64(v), to64(beta), C)
    check_T(to64(T_g), T_ref)
    check_WU(to64(W_g), W_ref, "bf16", "W")
    check_WU(to64(U_g), U_ref, "bf16", "U")
    assert np.isfinite(to64(T_g)).all()
