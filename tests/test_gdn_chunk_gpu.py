"""The chunk state recurrence and output (gdn_chunk_state_fwd) against the fp64 oracles (GPU).

Every call goes through the C ABI.  W and U~ come from the library's own kkt_solve on the same
inputs; the chunkwise oracle gets those very bf16 W and U~ (so it checks the consumer alone), and
the token-by-token recurrence oracle gets q, k, v, beta and g (so it checks the two kernels
together).  Tolerances: tests/compare.py.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import gdn
from gdn_chunkwise_ut_gb300 import _lib, chunk_gated_delta_rule, device_status, gdn_chunk_state_fwd, kkt_solve_fwd
from gdn_chunkwise_ut_gb300.inputs import make_gate, make_inputs, make_query, make_state, workloads
from tests.compare import check_recurrence, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
C = 64


def _case(B, T, H, cu=None, gated=False, h0=False, seed=0):
    k, v, beta = make_inputs(B, T, H, 128, 128, seed=seed, device=DEV)
    q = make_query(B, T, H, 128, seed=seed, device=DEV)
    g = make_gate(B, T, H, seed=seed, device=DEV) if gated else None
    N = B if cu is None else len(cu) - 1
    S0 = make_state(N, H, 128, 128, seed=seed, device=DEV) if h0 else None
    cu_t = None if cu is None else torch.as_tensor(np.asarray(cu), dtype=torch.int32, device=DEV)
    return q, k, v, beta, g, S0, cu_t


def _run(q, k, v, beta, g, S0, cu_t, scale=None):
    _, W, U = kkt_solve_fwd(k, v, beta, C, cu_t, materialize_T=False, g=g)
    o = torch.full(v.shape, float("nan"), device=DEV, dtype=torch.bfloat16)
    o, S = gdn_chunk_state_fwd(q, k, W, U, C, g=g, initial_state=S0, scale=scale, cu_seqlens=cu_t, o=o)
    torch.cuda.synchronize()
    assert device_status() == 0
    return W, U, o, S


def _check_both(q, k, v, beta, g, S0, cu_t, W, U, o, S, scale):
    cu = None if cu_t is None else cu_t.cpu().numpy()
    h0 = None if S0 is None else to64(S0)
    gg = None if g is None else to64(g)
    o_c, s_c = gdn.chunked_fwd(to64(q), to64(k), to64(W), to64(U), C, g=gg, initial_state=h0, scale=scale,
                               cu_seqlens=cu)
    a = check_recurrence(to64(o), o_c, to64(S), s_c, "chunkwise oracle: ")
    o_r, s_r = gdn.recurrent_fwd(to64(q), to64(k), to64(v), to64(beta), g=gg, initial_state=h0, scale=scale,
                                 cu_seqlens=cu)
    b = check_recurrence(to64(o), o_r, to64(S), s_r, "token recurrence: ")
    return a, b


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("h0", [False, True])
def test_fixed_length_ragged_tail(gated, h0):
    """Two sequences of 300 tokens (four chunks and a 44-token tail), three heads."""
    q, k, v, beta, g, S0, cu_t = _case(2, 300, 3, gated=gated, h0=h0, seed=11)
    W, U, o, S = _run(q, k, v, beta, g, S0, cu_t, scale=0.125)
    _check_both(q, k, v, beta, g, S0, cu_t, W, U, o, S, 0.125)


@pytest.mark.parametrize("gated", [False, True])
def test_varlen_with_empty_and_short_sequences(gated):
    """Packed sequences of 1, 63, 64, 65, 0, 130, 7 and 200 tokens, each with its own initial state;
    the empty sequence's final state is its initial state."""
    lengths = [1, 63, 64, 65, 0, 130, 7, 200]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    q, k, v, beta, g, S0, cu_t = _case(1, int(cu[-1]), 2, cu=cu, gated=gated, h0=True, seed=12)
    W, U, o, S = _run(q, k, v, beta, g, S0, cu_t)
    _check_both(q, k, v, beta, g, S0, cu_t, W, U, o, S, 128 ** -0.5)
    assert torch.equal(S[4], S0[4])


def test_no_tokens_copies_the_state():
    k = torch.zeros((2, 0, 3, 128), device=DEV, dtype=torch.bfloat16)
    S0 = make_state(2, 3, 128, 128, seed=5, device=DEV)
    o, S = gdn_chunk_state_fwd(k, k, k, k, C, initial_state=S0)
    torch.cuda.synchronize()
    assert o.numel() == 0 and torch.equal(S, S0)
    _, S = gdn_chunk_state_fwd(k, k, k, k, C)
    torch.cuda.synchronize()
    assert torch.count_nonzero(S).item() == 0


def test_unsupported_shapes_are_rejected():
    x = torch.zeros((1, 64, 1, 64), device=DEV, dtype=torch.bfloat16)
    o = torch.zeros_like(x)
    rc = _lib.lib().gdn_chunk_state_fwd(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), None, None, None,
                                        1, 64, 1, 64, 64, 64, 1.0, o.data_ptr(), None, None)
    assert rc == _lib.KKT_ERR_UNSUPPORTED
    y = torch.zeros((1, 64, 1, 128), device=DEV, dtype=torch.bfloat16)
    rc = _lib.lib().gdn_chunk_state_fwd(y.data_ptr(), y.data_ptr(), y.data_ptr(), y.data_ptr(), None, None, None,
                                        1, 64, 1, 128, 128, 32, 1.0, y.data_ptr(), None, None)
    assert rc == _lib.KKT_ERR_UNSUPPORTED


def test_malformed_cu_seqlens_is_reported_not_faulted():
    """A decreasing cu_seqlens: the kernel skips the bad sequences, records KKT_ERR_SEQLENS in the status
    word and leaves the context usable; a correct call right after matches the oracle."""
    q, k, v, beta, g, S0, _ = _case(1, 300, 2, seed=14)
    _, W, U = kkt_solve_fwd(k, v, beta, C)
    bad = torch.tensor([0, 200, 100, 300], dtype=torch.int32, device=DEV)
    gdn_chunk_state_fwd(q, k, W, U, C, cu_seqlens=bad)
    torch.cuda.synchronize()
    assert device_status() == _lib.KKT_ERR_SEQLENS
    assert device_status() == 0
    cu = np.array([0, 100, 300])
    cu_t = torch.as_tensor(cu, dtype=torch.int32, device=DEV)
    W, U, o, S = _run(q, k, v, beta, None, None, cu_t)
    _check_both(q, k, v, beta, None, None, cu_t, W, U, o, S, 128 ** -0.5)


def test_flashqla_signature_is_the_two_calls():
    """chunk_gated_delta_rule (the FlashQLA argument order) returns exactly kkt_solve then the
    chunk recurrence."""
    q, k, v, beta, g, S0, cu_t = _case(2, 200, 2, gated=True, h0=True, seed=13)
    o1, S1 = chunk_gated_delta_rule(q, k, v, g, beta, scale=0.2, initial_state=S0, output_final_state=True)
    _, _, o2, S2 = _run(q, k, v, beta, g, S0, cu_t, scale=0.2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


@pytest.mark.parametrize("name,gated", [("c2_t8192_h16", False), ("c3_b4_t8192_h16", False),
                                        ("c3_b4_t8192_h16", True), ("c4_varlen32_h32", False),
                                        ("c4_varlen32_h32", True), ("c5_b2_t16384_h24_c64", False)])
def test_full_size_every_element(name, gated):
    """A full-size workload: every element of o and of the final states against both oracles."""
    w = workloads()[name]
    k, v, beta, cu = w.make(seed=0, device=DEV)
    q = make_query(k.shape[0], k.shape[1], w.H, 128, seed=0, device=DEV)
    g = make_gate(k.shape[0], k.shape[1], w.H, seed=0, device=DEV) if gated else None
    N = w.B if cu is None else len(cu) - 1
    S0 = make_state(N, w.H, 128, 128, seed=0, device=DEV)
    cu_t = None if cu is None else torch.as_tensor(cu, dtype=torch.int32, device=DEV)
    W, U, o, S = _run(q, k, v, beta, g, S0, cu_t)
    _check_both(q, k, v, beta, g, S0, cu_t, W, U, o, S, 128 ** -0.5)
