"""Pins of the GDN recurrence oracle (oracle/gdn_oracle.c) to what the mathematics fixes.

Each pin takes the oracle library (so the mutation tests can run the same pins on planted mistakes)
and raises AssertionError when the oracle disagrees with:
  * the delta rule's defining property: right after a token with beta = 1 and a unit key, the
    state returns that token's value under its key (S_t^T k_t = v_t), with or without decay;
  * beta = 0 (nothing written): the state only decays, S_t = e^{g_1 + ... + g_t} S_0, and the
    output is scale * S_t^T q_t, in closed form;
  * orthogonal unit keys without decay: the erase factors commute, so the final state is
    (I - sum beta_i k_i k_i^T) S_0 + sum beta_i k_i v_i^T whatever the token order;
  * a token with zero decay (g = -1000) forgets everything before it;
  * linearity of the state and the output in (S_0, V) jointly;
  * a sequence split in two with the state handed over gives the unsplit result;
  * g = 0 is the ungated recurrence, bit for bit;
  * varlen batches equal per-sequence runs, each with its own initial state;
  * the chunkwise form fed with kkt_solve's W and U~ from the kkt oracle equals the token
    recurrence, for C in {1, 16, 32, 64}, gated or not, fixed length or varlen, with a ragged tail.
"""
from __future__ import annotations

import numpy as np

import oracle
from oracle import gdn


def _inputs(rng, B, T, H, dk, dv, gated=True):
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    beta = rng.uniform(0.05, 0.95, (B, T, H))
    g = rng.uniform(-0.4, 0.0, (B, T, H)) if gated else None
    return q, k, v, beta, g


def pin_retrieval_after_full_write(lib):
    """beta_t = 1 and ||k_t|| = 1: o_t with q_t = k_t, scale 1, is v_t (the delta rule replaces the
    value stored under k_t), whatever the earlier state and the decay."""
    rng = np.random.default_rng(50)
    q, k, v, beta, g = _inputs(rng, 1, 40, 2, 16, 8)
    beta[0, 17] = 1.0
    beta[0, 39] = 1.0
    q[0, 17] = k[0, 17]
    q[0, 39] = k[0, 39]
    h0 = rng.standard_normal((1, 2, 16, 8))
    for gg in (None, g):
        o, _ = gdn.recurrent_fwd(q, k, v, beta, g=gg, initial_state=h0, scale=1.0, lib=lib)
        np.testing.assert_allclose(o[0, 17], v[0, 17], atol=1e-12, rtol=0)
        np.testing.assert_allclose(o[0, 39], v[0, 39], atol=1e-12, rtol=0)


def pin_beta_zero_only_decays(lib):
    """beta = 0: S_t = e^{g_1 + ... + g_t} S_0 and o_t = scale S_t^T q_t."""
    rng = np.random.default_rng(51)
    q, k, v, beta, g = _inputs(rng, 2, 30, 2, 8, 4)
    beta[:] = 0.0
    h0 = rng.standard_normal((2, 2, 8, 4))
    o, ht = gdn.recurrent_fwd(q, k, v, beta, g=g, initial_state=h0, scale=0.3, lib=lib)
    G = np.cumsum(g, axis=1)                                   # [B, T, H]
    expect_o = 0.3 * np.exp(G)[..., None] * np.einsum("bthd,bhde->bthe", q, h0)
    np.testing.assert_allclose(o, expect_o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(ht, np.exp(G[:, -1])[..., None, None] * h0, atol=1e-12, rtol=0)


def pin_orthogonal_keys_closed_form(lib):
    """Orthogonal unit keys, no decay: S_L = (I - sum beta k k^T) S_0 + sum beta k v^T, and the
    result does not depend on the order of the tokens."""
    rng = np.random.default_rng(52)
    L, dk, dv = 12, 16, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm[:L].reshape(1, L, 1, dk)
    v = rng.standard_normal((1, L, 1, dv))
    beta = rng.uniform(0.05, 0.95, (1, L, 1))
    q = rng.standard_normal((1, L, 1, dk))
    h0 = rng.standard_normal((1, 1, dk, dv))
    _, ht = gdn.recurrent_fwd(q, k, v, beta, initial_state=h0, lib=lib)
    K, V, b = k[0, :, 0], v[0, :, 0], beta[0, :, 0]
    expect = (np.eye(dk) - (K.T * b) @ K) @ h0[0, 0] + (K.T * b) @ V
    np.testing.assert_allclose(ht[0, 0], expect, atol=1e-12, rtol=0)
    perm = rng.permutation(L)
    _, ht2 = gdn.recurrent_fwd(q[:, perm], k[:, perm], v[:, perm], beta[:, perm], initial_state=h0, lib=lib)
    np.testing.assert_allclose(ht2, ht, atol=1e-12, rtol=0)


def pin_zero_decay_forgets(lib):
    """A token with g = -1000 (alpha underflows to 0) drops every earlier contribution: the run equals
    a run started at that token from a zero state."""
    rng = np.random.default_rng(53)
    q, k, v, beta, g = _inputs(rng, 1, 50, 2, 8, 8)
    g[0, 20, :] = -1000.0
    h0 = rng.standard_normal((1, 2, 8, 8))
    o, ht = gdn.recurrent_fwd(q, k, v, beta, g=g, initial_state=h0, lib=lib)
    o2, ht2 = gdn.recurrent_fwd(q[:, 20:], k[:, 20:], v[:, 20:], beta[:, 20:], g=g[:, 20:], lib=lib)
    np.testing.assert_allclose(o[:, 20:], o2, atol=1e-12, rtol=0)
    np.testing.assert_allclose(ht, ht2, atol=1e-12, rtol=0)


def pin_linear_in_state_and_values(lib):
    """The state and output are linear in (S_0, V) jointly (k, beta, g, q fixed)."""
    rng = np.random.default_rng(54)
    q, k, v, beta, g = _inputs(rng, 1, 37, 2, 8, 4)
    v2 = rng.standard_normal(v.shape)
    h0, h02 = rng.standard_normal((2, 1, 2, 8, 4))
    a, b = 0.7, -1.3
    o1, s1 = gdn.recurrent_fwd(q, k, v, beta, g=g, initial_state=h0, scale=0.5, lib=lib)
    o2, s2 = gdn.recurrent_fwd(q, k, v2, beta, g=g, initial_state=h02, scale=0.5, lib=lib)
    o3, s3 = gdn.recurrent_fwd(q, k, a * v + b * v2, beta, g=g, initial_state=a * h0 + b * h02, scale=0.5, lib=lib)
    np.testing.assert_allclose(o3, a * o1 + b * o2, atol=1e-11, rtol=0)
    np.testing.assert_allclose(s3, a * s1 + b * s2, atol=1e-11, rtol=0)
    # and not linear in q's scale alone through the state: scale multiplies the output only
    o4, s4 = gdn.recurrent_fwd(q, k, v, beta, g=g, initial_state=h0, scale=1.0, lib=lib)
    np.testing.assert_allclose(o4, 2.0 * o1, atol=1e-12, rtol=0)
    np.testing.assert_array_equal(s4, s1)


def pin_split_hands_over_state(lib):
    """Tokens 0..m-1 then m..L-1 with the first part's final state as the second part's initial state
    equal the unsplit run."""
    rng = np.random.default_rng(55)
    q, k, v, beta, g = _inputs(rng, 2, 45, 3, 8, 8)
    h0 = rng.standard_normal((2, 3, 8, 8))
    o, ht = gdn.recurrent_fwd(q, k, v, beta, g=g, initial_state=h0, lib=lib)
    m = 19
    oa, ha = gdn.recurrent_fwd(q[:, :m], k[:, :m], v[:, :m], beta[:, :m], g=g[:, :m], initial_state=h0, lib=lib)
    ob, hb = gdn.recurrent_fwd(q[:, m:], k[:, m:], v[:, m:], beta[:, m:], g=g[:, m:], initial_state=ha, lib=lib)
    np.testing.assert_allclose(np.concatenate([oa, ob], axis=1), o, atol=1e-13, rtol=0)
    np.testing.assert_allclose(hb, ht, atol=1e-13, rtol=0)


def pin_gate_zero_is_ungated(lib):
    rng = np.random.default_rng(56)
    q, k, v, beta, _ = _inputs(rng, 1, 33, 2, 8, 4, gated=False)
    h0 = rng.standard_normal((1, 2, 8, 4))
    a = gdn.recurrent_fwd(q, k, v, beta, initial_state=h0, lib=lib)
    b = gdn.recurrent_fwd(q, k, v, beta, g=np.zeros(beta.shape), initial_state=h0, lib=lib)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    W = oracle.oracle_fwd(k, v, beta, 16)[1]
    U = oracle.oracle_fwd(k, v, beta, 16)[2]
    c = gdn.chunked_fwd(q, k, W, U, 16, initial_state=h0, lib=lib)
    d = gdn.chunked_fwd(q, k, W, U, 16, g=np.zeros(beta.shape), initial_state=h0, lib=lib)
    for x, y in zip(c, d):
        np.testing.assert_array_equal(x, y)


def pin_varlen_equals_per_sequence(lib):
    """Packed sequences equal per-sequence runs, each from its own initial state (both forms)."""
    rng = np.random.default_rng(57)
    cu = np.array([0, 7, 7, 70, 71, 130])
    N = int(cu[-1])
    q, k, v, beta, g = _inputs(rng, 1, N, 2, 8, 4)
    h0 = rng.standard_normal((len(cu) - 1, 2, 8, 4))
    o, ht = gdn.recurrent_fwd(q, k, v, beta, g=g, initial_state=h0, cu_seqlens=cu, lib=lib)
    _, W, U = oracle.oracle_fwd(k, v, beta, 32, cu_seqlens=cu, g=g)
    oc, hc = gdn.chunked_fwd(q, k, W, U, 32, g=g, initial_state=h0, cu_seqlens=cu, lib=lib)
    for s in range(len(cu) - 1):
        a, e = int(cu[s]), int(cu[s + 1])
        sl = lambda x: x[:, a:e]
        os_, hs = gdn.recurrent_fwd(sl(q), sl(k), sl(v), sl(beta), g=sl(g), initial_state=h0[s:s + 1], lib=lib)
        np.testing.assert_array_equal(o[:, a:e], os_)
        np.testing.assert_array_equal(ht[s:s + 1], hs)
        np.testing.assert_allclose(oc[:, a:e], os_, atol=1e-12, rtol=0)
        np.testing.assert_allclose(hc[s:s + 1], hs, atol=1e-12, rtol=0)


def pin_chunked_equals_recurrent(lib):
    """The chunkwise form from kkt_solve's W and U~ (the kkt oracle's) reproduces the token recurrence:
    every chunk size, gated and not, a ragged tail, a nonzero initial state."""
    rng = np.random.default_rng(58)
    B, T, H, dk, dv = 2, 150, 2, 16, 8
    for gated in (False, True):
        q, k, v, beta, g = _inputs(rng, B, T, H, dk, dv, gated=gated)
        h0 = rng.standard_normal((B, H, dk, dv))
        o, ht = gdn.recurrent_fwd(q, k, v, beta, g=g, initial_state=h0, scale=0.25)
        for C in (1, 16, 32, 64):
            _, W, U = oracle.oracle_fwd(k, v, beta, C, g=g)
            oc, hc = gdn.chunked_fwd(q, k, W, U, C, g=g, initial_state=h0, scale=0.25, lib=lib)
            np.testing.assert_allclose(oc, o, atol=1e-11, rtol=0)
            np.testing.assert_allclose(hc, ht, atol=1e-11, rtol=0)


RECURRENT_PINS = [
    pin_retrieval_after_full_write,
    pin_beta_zero_only_decays,
    pin_orthogonal_keys_closed_form,
    pin_zero_decay_forgets,
    pin_linear_in_state_and_values,
    pin_split_hands_over_state,
    pin_gate_zero_is_ungated,
    pin_varlen_equals_per_sequence,
]

PINS = RECURRENT_PINS + [pin_chunked_equals_recurrent]
