"""kkt_solve_fwd_host, the C ABI's host-buffer entry point (GPU): the pipelined copies in, kernels and
copies out give exactly what one device call gives, for any number of pieces, fixed-length and
varlen batches, the gated variant, fp16 T, no T, and pageable host memory; and the oracle agrees."""
import numpy as np
import pytest
import torch

from gdn_chunkwise_ut_gb300 import device_status, kkt_solve_fwd
from gdn_chunkwise_ut_gb300.api import host_workspace_bytes, kkt_solve_fwd_host
from gdn_chunkwise_ut_gb300.inputs import make_gate, make_inputs
from tests.test_parity_gpu import full_compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _host(x, pinned=True):
    return None if x is None else (x.cpu().pin_memory() if pinned else x.cpu())


@pytest.mark.parametrize("pieces", [1, 3, 8, 64])
@pytest.mark.parametrize("C", [32, 64, 128])
def test_fixed_length_any_pieces(C, pieces):
    k, v, beta = make_inputs(3, 1000, 5, 128, 128, seed=200 + C, device=DEV)
    ref = kkt_solve_fwd(k, v, beta, C)
    torch.cuda.synchronize()
    outs = kkt_solve_fwd_host(_host(k), _host(v), _host(beta), C, pieces=pieces)
    for a, b in zip(ref, outs):
        assert torch.equal(a.cpu(), b)
    assert device_status() == 0
    if pieces == 8:
        full_compare(k, v, beta, C, None, tuple(x.to(DEV) for x in outs))


@pytest.mark.parametrize("pieces", [1, 4, 9])
def test_varlen_gated_fp16(pieces):
    lengths = [1, 63, 64, 0, 700, 130, 7, 1200, 5, 0, 66]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    k, v, beta = make_inputs(1, int(cu[-1]), 3, 128, 128, seed=210, device=DEV)
    g = make_gate(1, int(cu[-1]), 3, seed=210, device=DEV)
    cu_d = torch.as_tensor(cu, device=DEV)
    for C in (64, 128):
        ref = kkt_solve_fwd(k, v, beta, C, cu_d, g=g, T_dtype=torch.float16)
        torch.cuda.synchronize()
        outs = kkt_solve_fwd_host(_host(k), _host(v), _host(beta), C, list(cu), g=_host(g), T_dtype=torch.float16,
                                  pieces=pieces)
        for a, b in zip(ref, outs):
            assert torch.equal(a.cpu(), b)
    assert device_status() == 0


def test_no_T_pageable_memory_and_workspace_reuse():
    k, v, beta = make_inputs(2, 777, 4, 64, 128, seed=220, device=DEV)
    ref = kkt_solve_fwd(k, v, beta, 64, materialize_T=False)
    torch.cuda.synchronize()
    ws = torch.empty(host_workspace_bytes(2, 777, 4, 64, 128, 64, pieces=5), dtype=torch.uint8, device=DEV)
    for _ in range(2):  # the second call reuses the workspace; the inputs are pageable
        outs = kkt_solve_fwd_host(_host(k, False), _host(v, False), _host(beta, False), 64, materialize_T=False,
                                  pieces=5, workspace=ws)
        assert outs[0] is None
        for a, b in zip(ref[1:], outs[1:]):
            assert torch.equal(a.cpu(), b)
    assert device_status() == 0


def test_ordered_on_the_callers_stream():
    """Issued on a side stream without waiting: work queued after it on that stream sees the
    outputs, and a second call with other inputs does not disturb the first call's results."""
    k, v, beta = make_inputs(2, 2000, 4, 128, 128, seed=230, device=DEV)
    k2, v2, beta2 = make_inputs(2, 2000, 4, 128, 128, seed=231, device=DEV)
    ref = kkt_solve_fwd(k, v, beta, 64)
    ref2 = kkt_solve_fwd(k2, v2, beta2, 64)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    hosts = [_host(x) for x in (k, v, beta)]
    hosts2 = [_host(x) for x in (k2, v2, beta2)]
    out1 = kkt_solve_fwd_host(*hosts, 64, pieces=6, stream=s, sync=False)
    out2 = kkt_solve_fwd_host(*hosts2, 64, pieces=6, stream=s, sync=False)
    s.synchronize()
    for a, b in zip(ref, out1):
        assert torch.equal(a.cpu(), b)
    for a, b in zip(ref2, out2):
        assert torch.equal(a.cpu(), b)
    assert device_status() == 0
