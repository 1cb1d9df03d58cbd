"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each pin takes a loaded oracle library (``oracle.load()`` or a mutant build)
and raises AssertionError when the oracle disagrees with:
  * a chunk worked by hand from the definitions (tests/golden/closed_form_c3.json),
  * exact rational brute force on tiny chunks (fractions.Fraction),
  * the inverse invariant T A = I and exact unit-lower-triangularity,
  * a library inverse / solve (numpy.linalg) on the oracle's coefficient matrix,
  * an independent fp64 blocked recursion and the 2x2 block-inverse identity,
  * the degenerate cases the page asks for (beta = 0; only the sub-diagonal
    block nonzero) and orthogonal keys,
  * causality of the chunk (a short last chunk equals the top-left block of a
    full one), the varlen/fixed-length equivalence and the tensor layout,
  * the page's measured cond(A) bounds,
  * the gated coefficient diag(beta)(Gamma o K K^T) (§5 item 12): no decay is the
    ungated oracle; the page's two differently scaled copies of K; any gate is a
    diagonal similarity of the ungated matrix, so T = Gamma o T0 and W = diag(e^G) W0
    (the keys of W carry the decay from the chunk's start); a token with zero
    decay cuts the chunk into independent blocks; the tensor layout of the gate.
Sources: "TileLang 实战：单位下三角矩阵求逆" §1, §2.1, §2.2, §2.4, §3.2, §4, §5.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand_chunk(rng, Lc, dk, dv):
    k = rng.standard_normal((Lc, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((Lc, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(Lc)))
    return k, v, beta


def _hadamard16():
    h = np.array([[1.0]])
    for _ in range(4):
        h = np.block([[h, h], [h, -h]])
    return h


# --- hand-worked and brute-force values -------------------------------------------------

def pin_closed_form_c3(lib):
    """Three tokens worked by hand (§1 definitions, §3.2 beta on rows, unit diagonal)."""
    with open(os.path.join(GOLDEN, "closed_form_c3.json")) as f:
        g = json.load(f)
    for C in (3, 4, 16):  # also as the short last chunk of a wider chunk
        T, W, U, A = oracle.oracle_chunk(g["k"], g["v"], g["beta"], C, lib=lib)
        np.testing.assert_allclose(A[:3, :3], g["A"], atol=1e-15, rtol=0)
        np.testing.assert_allclose(T[:, :3], g["T"], atol=1e-15, rtol=0)
        assert np.all(T[:, 3:] == 0.0)
        np.testing.assert_allclose(W, g["W"], atol=1e-15, rtol=0)
        np.testing.assert_allclose(U, g["U"], atol=1e-15, rtol=0)


def _exact_reference(k, v, beta):
    """Exact rational A, T = A^-1 (Gauss-Jordan), W = T diag(beta) K, U = T diag(beta) V."""
    n = len(beta)
    kf = [[Fraction(x) for x in row] for row in k]
    vf = [[Fraction(x) for x in row] for row in v]
    bf = [Fraction(x) for x in beta]
    A = [[Fraction(0)] * n for _ in range(n)]
    for i in range(n):
        for j in range(n):
            if i == j:
                A[i][j] = Fraction(1)
            elif i > j:
                A[i][j] = bf[i] * sum(a * b for a, b in zip(kf[i], kf[j]))
    aug = [A[i][:] + [Fraction(int(i == j)) for j in range(n)] for i in range(n)]
    for c in range(n):
        p = aug[c][c]
        aug[c] = [x / p for x in aug[c]]
        for r in range(n):
            if r != c and aug[r][c] != 0:
                f = aug[r][c]
                aug[r] = [x - f * y for x, y in zip(aug[r], aug[c])]
    T = [row[n:] for row in aug]
    W = [[sum(T[i][j] * bf[j] * kf[j][e] for j in range(n)) for e in range(len(kf[0]))] for i in range(n)]
    U = [[sum(T[i][j] * bf[j] * vf[j][e] for j in range(n)) for e in range(len(vf[0]))] for i in range(n)]
    to = lambda m: np.array([[float(x) for x in row] for row in m])
    return to(A), to(T), to(W), to(U)


def pin_exact_rational_bruteforce(lib):
    """Exact rational Gauss-Jordan on dyadic inputs; every entry of A nonzero."""
    rng = np.random.default_rng(7)
    for n, dk, dv in ((5, 3, 2), (7, 4, 3)):
        k = rng.integers(-8, 9, (n, dk)) / 8.0
        v = rng.integers(-8, 9, (n, dv)) / 8.0
        beta = rng.integers(1, 16, n) / 16.0
        A_x, T_x, W_x, U_x = _exact_reference(k, v, beta)
        T, W, U, A = oracle.oracle_chunk(k, v, beta, n, lib=lib)
        np.testing.assert_allclose(A, A_x, atol=1e-13, rtol=0)
        np.testing.assert_allclose(T, T_x, atol=1e-12, rtol=1e-13)
        np.testing.assert_allclose(W, W_x, atol=1e-12, rtol=1e-13)
        np.testing.assert_allclose(U, U_x, atol=1e-12, rtol=1e-13)


# --- invariants and library cross-checks -------------------------------------------------

def pin_inverse_invariant(lib):
    """T A = I to 1e-12, T exactly unit lower triangular (§2.1)."""
    rng = np.random.default_rng(11)
    for C in (16, 32, 64, 128):
        k, v, beta = _rand_chunk(rng, C, 128, 128)
        T, W, U, A = oracle.oracle_chunk(k, v, beta, C, lib=lib)
        assert np.abs(T @ A - np.eye(C)).max() <= 1e-12
        assert np.all(np.diag(T) == 1.0)
        assert np.all(np.triu(T, 1) == 0.0)
        assert np.all(np.diag(A) == 1.0) and np.all(np.triu(A, 1) == 0.0)


def pin_library_inverse_and_solve(lib):
    """numpy.linalg.inv(A) and solve(A, diag(beta) K) agree (§4 compares against np.linalg.inv)."""
    rng = np.random.default_rng(12)
    with open(os.path.join(GOLDEN, "paper_counts.json")) as f:
        errs = json.load(f)["inverse_errors"]
    worst = 0.0
    for C in (16, 32, 64):
        for _ in range(10):
            k, v, beta = _rand_chunk(rng, C, 128, 64)
            T, W, U, A = oracle.oracle_chunk(k, v, beta, C, lib=lib)
            worst = max(worst, np.abs(T - np.linalg.inv(A)).max())
            np.testing.assert_allclose(W, np.linalg.solve(A, beta[:, None] * k), atol=1e-13, rtol=0)
            np.testing.assert_allclose(U, np.linalg.solve(A, beta[:, None] * v), atol=1e-13, rtol=0)
            assert np.abs(A @ W - beta[:, None] * k).max() <= 1e-12
    # the page's own numpy mirror reaches 2.22e-15 on a 16x16 row substitution
    assert worst <= errs["row16"], worst


def _blocked_inverse(L, base=16):
    """Independent fp64 recursion of §2.2: [[L00^-1, 0], [-L11^-1 L10 L00^-1, L11^-1]]."""
    n = L.shape[0]
    if n <= base:
        return np.linalg.inv(L)
    h = n // 2
    i00 = _blocked_inverse(L[:h, :h], base)
    i11 = _blocked_inverse(L[h:, h:], base)
    out = np.zeros_like(L)
    out[:h, :h] = i00
    out[h:, h:] = i11
    out[h:, :h] = -i11 @ L[h:, :h] @ i00
    return out


def pin_block_inverse_identity(lib):
    """The 2x2 block-inverse identity of §2.2 and its check L10 L00^-1 + L11 T10 = 0."""
    rng = np.random.default_rng(13)
    for C in (32, 64, 128):
        k, v, beta = _rand_chunk(rng, C, 128, 32)
        T, W, U, A = oracle.oracle_chunk(k, v, beta, C, lib=lib)
        np.testing.assert_allclose(T, _blocked_inverse(A), atol=1e-13, rtol=0)
        h = C // 2
        L00, L10, L11 = A[:h, :h], A[h:, :h], A[h:, h:]
        assert np.abs(L10 @ T[:h, :h] + L11 @ T[h:, :h]).max() <= 1e-13
        np.testing.assert_allclose(T[:h, :h], np.linalg.inv(L00), atol=1e-13, rtol=0)
        np.testing.assert_allclose(T[h:, h:], np.linalg.inv(L11), atol=1e-13, rtol=0)


# --- degenerate cases ---------------------------------------------------------------------

def pin_beta_zero(lib):
    """beta = 0 gives A = T = I and W = U = 0 (§4, first mandatory degenerate test)."""
    rng = np.random.default_rng(14)
    k, v, _ = _rand_chunk(rng, 32, 64, 64)
    T, W, U, A = oracle.oracle_chunk(k, v, np.zeros(32), 32, lib=lib)
    assert np.array_equal(T, np.eye(32)) and np.array_equal(A, np.eye(32))
    assert np.all(W == 0.0) and np.all(U == 0.0)


def pin_orthogonal_keys(lib):
    """Mutually orthogonal keys: S = 0 below the diagonal, so T = I, W = diag(beta) K."""
    rng = np.random.default_rng(15)
    perm = rng.permutation(32)
    k = np.zeros((32, 32))
    k[np.arange(32), perm] = rng.choice([-1.0, 1.0], 32)
    v = rng.standard_normal((32, 16))
    beta = rng.uniform(0.05, 0.95, 32)
    T, W, U, A = oracle.oracle_chunk(k, v, beta, 32, lib=lib)
    assert np.array_equal(T, np.eye(32))
    np.testing.assert_array_equal(W, beta[:, None] * k)
    np.testing.assert_array_equal(U, beta[:, None] * v)


def subdiagonal_only_case(beta):
    """Keys for which only the 16x16 sub-diagonal block of A is nonzero.

    Rows 0..15 are the unit vectors e_0..e_15, rows 16..31 the rows of a
    16x16 Hadamard matrix scaled by 1/4 (orthonormal, every value exact in
    bf16).  Within each block the keys are orthonormal, so L00 = L11 = I; across
    blocks <k_i, k_j> = H[i-16, j] / 4, so L10[i, j] = beta_{16+i} H[i, j] / 4.
    """
    k = np.zeros((32, 32))
    k[:16, :16] = np.eye(16)
    k[16:, :16] = _hadamard16() / 4.0
    L10 = beta[16:, None] * _hadamard16() / 4.0
    return k, L10


def pin_subdiagonal_block_only(lib):
    """§4, second mandatory degenerate test: T's lower-left block is exactly -L10."""
    rng = np.random.default_rng(16)
    beta = rng.integers(1, 64, 32) / 64.0  # distinct row scales expose beta on the wrong side
    k, L10 = subdiagonal_only_case(beta)
    v = rng.standard_normal((32, 8))
    T, W, U, A = oracle.oracle_chunk(k, v, beta, 32, lib=lib)
    np.testing.assert_array_equal(A[16:, :16], L10)
    np.testing.assert_array_equal(T[:16, :16], np.eye(16))
    np.testing.assert_array_equal(T[16:, 16:], np.eye(16))
    np.testing.assert_array_equal(T[16:, :16], -L10)
    assert np.all(T[:16, 16:] == 0.0)


# --- chunking, layout, varlen --------------------------------------------------------------

def pin_short_chunk_is_leading_block(lib):
    """A short last chunk equals the leading block of a full one (A is lower triangular)."""
    rng = np.random.default_rng(17)
    k, v, beta = _rand_chunk(rng, 64, 128, 96)
    Tf, Wf, Uf, _ = oracle.oracle_chunk(k, v, beta, 64, lib=lib)
    for Lc in (1, 7, 33, 63):
        T, W, U, _ = oracle.oracle_chunk(k[:Lc], v[:Lc], beta[:Lc], 64, lib=lib)
        np.testing.assert_allclose(T[:, :Lc], Tf[:Lc, :Lc], atol=1e-14, rtol=0)
        assert np.all(T[:, Lc:] == 0.0)
        np.testing.assert_allclose(W, Wf[:Lc], atol=1e-14, rtol=0)
        np.testing.assert_allclose(U, Uf[:Lc], atol=1e-14, rtol=0)


def pin_tensor_layout(lib):
    """Whole-tensor driver: token n, head h of chunk c equals the chunk computed alone."""
    rng = np.random.default_rng(18)
    B, T, H, dk, dv, C = 2, 70, 3, 16, 8, 32
    k = rng.standard_normal((B, T, H, dk)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    beta = rng.uniform(0.05, 0.95, (B, T, H))
    To, Wo, Uo = oracle.oracle_fwd(k, v, beta, C, lib=lib)
    for b in range(B):
        for h in range(H):
            for t0 in range(0, T, C):
                t1 = min(T, t0 + C)
                Tc, Wc, Uc, _ = oracle.oracle_chunk(k[b, t0:t1, h], v[b, t0:t1, h], beta[b, t0:t1, h], C, lib=lib)
                np.testing.assert_array_equal(To[b, t0:t1, h], Tc)
                np.testing.assert_array_equal(Wo[b, t0:t1, h], Wc)
                np.testing.assert_array_equal(Uo[b, t0:t1, h], Uc)


def pin_varlen_equals_fixed(lib):
    """Packed sequences give the rows each sequence gives on its own."""
    rng = np.random.default_rng(19)
    lengths = [5, 64, 100, 1, 33]
    H, dk, dv, C = 2, 16, 16, 32
    cu = np.concatenate([[0], np.cumsum(lengths)])
    k = rng.standard_normal((1, cu[-1], H, dk)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, cu[-1], H, dv))
    beta = rng.uniform(0.05, 0.95, (1, cu[-1], H))
    To, Wo, Uo = oracle.oracle_fwd(k, v, beta, C, cu_seqlens=cu, lib=lib)
    for s, L in enumerate(lengths):
        a, b = cu[s], cu[s + 1]
        Ts, Ws, Us = oracle.oracle_fwd(k[:, a:b], v[:, a:b], beta[:, a:b], C, lib=lib)
        np.testing.assert_array_equal(To[:, a:b], Ts)
        np.testing.assert_array_equal(Wo[:, a:b], Ws)
        np.testing.assert_array_equal(Uo[:, a:b], Us)


def pin_cond_bounds(lib):
    """cond_2(A) stays under the page's measured bounds (§2.4 second table) at d_k = 128."""
    with open(os.path.join(GOLDEN, "paper_counts.json")) as f:
        bounds = json.load(f)["cond_upper_bound"]["values"]
    rng = np.random.default_rng(20)
    for C in (32, 64, 128):
        worst = 0.0
        for _ in range(200):
            k, v, beta = _rand_chunk(rng, C, 128, 1)
            _, _, _, A = oracle.oracle_chunk(k, v, beta, C, lib=lib)
            worst = max(worst, np.linalg.cond(A))
        assert worst <= bounds[str(C)], (C, worst)


# --- the gated coefficient ------------------------------------------------------------------

def pin_gate_zero_is_ungated(lib):
    """g = 0 (decay alpha = 1 everywhere): the gated oracle is the ungated one, bit for bit."""
    rng = np.random.default_rng(30)
    k, v, beta = _rand_chunk(rng, 50, 32, 16)
    ref = oracle.oracle_chunk(k, v, beta, 64, lib=lib)
    got = oracle.oracle_chunk(k, v, beta, 64, lib=lib, g=np.zeros(50))
    for a, b in zip(ref, got):
        np.testing.assert_array_equal(a, b)


def pin_gate_two_scaled_keys(lib):
    """The gated A is I + strictLower((diag(beta e^G) K)(diag(e^-G) K)^T), G the prefix sums of
    the chunk's log decays: the two differently scaled copies of K of §5 item 12."""
    rng = np.random.default_rng(31)
    for Lc, C in ((64, 64), (40, 64), (128, 128), (9, 32)):
        k, v, beta = _rand_chunk(rng, Lc, 32, 8)
        g = rng.uniform(-0.2, 0.0, Lc)
        G = np.cumsum(g)
        left = (beta * np.exp(G))[:, None] * k
        right = np.exp(-G)[:, None] * k
        _, _, _, A = oracle.oracle_chunk(k, v, beta, C, lib=lib, g=g)
        expect = np.eye(C)
        expect[:Lc, :Lc] += np.tril(left @ right.T, -1)
        np.testing.assert_allclose(A, expect, atol=1e-13, rtol=0)


def pin_gate_similarity(lib):
    """Gamma[i][j] = e^{G_i - G_j} makes the gated A a diagonal similarity of the ungated one,
    A = D A0 D^-1 with D = diag(e^{G_i}), so T = D T0 D^-1: T[i][j] = e^{G_i - G_j} T0[i][j] with T0
    the ungated inverse, for any gate (a constant one, e^{c (i - j)}, and a random one).  The keys
    of W carry the decay from the chunk's start, gamma = e^G, so W = T diag(beta gamma) K, which by
    the same similarity is D T0 diag(beta) K = diag(gamma) W0 with W0 the ungated W; U~ =
    T diag(beta) V."""
    rng = np.random.default_rng(32)
    Lc, C = 48, 64
    k, v, beta = _rand_chunk(rng, Lc, 32, 16)
    T0, W0, _, _ = oracle.oracle_chunk(k, v, beta, C, lib=lib)
    for g in (np.full(Lc, -0.15), rng.uniform(-0.4, 0.0, Lc)):
        T, W, U, _ = oracle.oracle_chunk(k, v, beta, C, lib=lib, g=g)
        G = np.cumsum(g)
        expect = T0[:, :Lc] * np.exp(G[:, None] - G[None, :])
        np.testing.assert_allclose(T[:, :Lc], expect, atol=1e-13, rtol=0)
        assert np.all(T[:, Lc:] == 0.0)
        np.testing.assert_allclose(W, expect @ ((beta * np.exp(G))[:, None] * k), atol=1e-12, rtol=0)
        np.testing.assert_allclose(W, np.exp(G)[:, None] * W0, atol=1e-12, rtol=0)
        np.testing.assert_allclose(U, expect @ (beta[:, None] * v), atol=1e-12, rtol=0)


def pin_gate_cut_decouples(lib):
    """A token whose decay is zero (g_c = -1000: exp underflows to 0) cuts the chunk: Gamma[i][j] = 0
    for j < c <= i, so T is block diagonal; the leading block is the chunk of tokens 0..c-1 alone and
    the trailing block the chunk of tokens c.. alone (g_c itself enters no product there)."""
    rng = np.random.default_rng(33)
    Lc, C, cut = 60, 64, 23
    k, v, beta = _rand_chunk(rng, Lc, 32, 16)
    g = rng.uniform(-0.3, 0.0, Lc)
    g[cut] = -1000.0
    T, W, U, _ = oracle.oracle_chunk(k, v, beta, C, lib=lib, g=g)
    T1, W1, U1, _ = oracle.oracle_chunk(k[:cut], v[:cut], beta[:cut], C, lib=lib, g=g[:cut])
    T2, W2, U2, _ = oracle.oracle_chunk(k[cut:], v[cut:], beta[cut:], C, lib=lib, g=g[cut:])
    assert np.all(T[cut:, :cut] == 0.0) and np.all(T[:cut, cut:] == 0.0)
    np.testing.assert_allclose(T[:cut, :cut], T1[:, :cut], atol=1e-14, rtol=0)
    np.testing.assert_allclose(T[cut:, cut:Lc], T2[:, :Lc - cut], atol=1e-14, rtol=0)
    for X, X1, X2 in ((W, W1, W2), (U, U1, U2)):
        np.testing.assert_allclose(X[:cut], X1, atol=1e-14, rtol=0)
        np.testing.assert_allclose(X[cut:], X2, atol=1e-14, rtol=0)


def pin_gate_tensor_layout(lib):
    """Whole-tensor driver with a gate: token n, head h of chunk c equals the chunk computed alone
    with that chunk's own gates (the gate restarts at every chunk), fixed length and varlen."""
    rng = np.random.default_rng(34)
    B, T, H, dk, dv, C = 2, 70, 3, 16, 8, 32
    k = rng.standard_normal((B, T, H, dk)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    beta = rng.uniform(0.05, 0.95, (B, T, H))
    g = rng.uniform(-0.5, 0.0, (B, T, H))
    To, Wo, Uo = oracle.oracle_fwd(k, v, beta, C, lib=lib, g=g)
    for b in range(B):
        for h in range(H):
            for t0 in range(0, T, C):
                t1 = min(T, t0 + C)
                Tc, Wc, Uc, _ = oracle.oracle_chunk(k[b, t0:t1, h], v[b, t0:t1, h], beta[b, t0:t1, h], C,
                                                    lib=lib, g=g[b, t0:t1, h])
                np.testing.assert_array_equal(To[b, t0:t1, h], Tc)
                np.testing.assert_array_equal(Wo[b, t0:t1, h], Wc)
                np.testing.assert_array_equal(Uo[b, t0:t1, h], Uc)
    cu = [0, 20, 20, 101, 140]
    kf, vf, bf, gf = (x.reshape((1, B * T) + x.shape[2:]) for x in (k, v, beta, g))
    To, Wo, Uo = oracle.oracle_fwd(kf, vf, bf, C, cu_seqlens=cu, lib=lib, g=gf)
    for s in range(len(cu) - 1):
        a, e = cu[s], cu[s + 1]
        Ts, Ws, Us = oracle.oracle_fwd(kf[:, a:e], vf[:, a:e], bf[:, a:e], C, lib=lib, g=gf[:, a:e])
        np.testing.assert_array_equal(To[:, a:e], Ts)
        np.testing.assert_array_equal(Wo[:, a:e], Ws)
        np.testing.assert_array_equal(Uo[:, a:e], Us)


PINS = [
    pin_closed_form_c3,
    pin_exact_rational_bruteforce,
    pin_inverse_invariant,
    pin_library_inverse_and_solve,
    pin_block_inverse_identity,
    pin_beta_zero,
    pin_orthogonal_keys,
    pin_subdiagonal_block_only,
    pin_short_chunk_is_leading_block,
    pin_tensor_layout,
    pin_varlen_equals_fixed,
    pin_cond_bounds,
    pin_gate_zero_is_ungated,
    pin_gate_two_scaled_keys,
    pin_gate_similarity,
    pin_gate_cut_decouples,
    pin_gate_tensor_layout,
]
