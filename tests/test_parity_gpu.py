"""CUDA path against the fp64 oracle, element by element (GPU).

Every call goes through the C ABI (libkkt.so via the ctypes binding).  These are
the small and edge cases, compared in full; the full-size workloads are compared
element by element in tests/test_full_size_gpu.py.
"""
import numpy as np
import pytest
import torch

import oracle
from gdn_chunkwise_ut_gb300 import _lib, device_status, kkt_solve_fwd, select_kernel
from gdn_chunkwise_ut_gb300.inputs import make_gate, make_inputs, workloads
from tests.compare import check_T, check_WU, chunks, to64
from tests.pins import subdiagonal_only_case

pytestmark = pytest.mark.gpu
DEV = "cuda"


def kernels_for(dk, dv, C, io="bf16"):
    out = []
    for kern in ("simt", "tc"):
        try:
            select_kernel(dk, dv, C, io, kern)
            out.append(kern)
        except _lib.KktError:
            pass
    return out


ALL_KERNELS = ["simt", "tc"]


def _skip_unless(kernel, dk, dv, C, io="bf16"):
    if kernel not in kernels_for(dk, dv, C, io):
        pytest.skip(f"{kernel} kernel does not cover dk={dk} dv={dv} C={C} io={io}")


def run(k, v, beta, C, cu=None, kernel="auto", poison=True, workspace="auto", g=None):
    """Calls the library with NaN-poisoned outputs; returns (T, W, U) on the device."""
    Bt, T, H, dk = k.shape
    dv = v.shape[-1]
    T_out = torch.full((Bt, T, H, C), float("nan"), device=DEV)
    W = torch.full((Bt, T, H, dk), float("nan"), device=DEV, dtype=k.dtype)
    U = torch.full((Bt, T, H, dv), float("nan"), device=DEV, dtype=k.dtype)
    cu_t = None if cu is None else torch.as_tensor(np.asarray(cu), dtype=torch.int32, device=DEV)
    kkt_solve_fwd(k, v, beta, C, cu_t, T_out=T_out, W_out=W, U_out=U, kernel=kernel, workspace=workspace, g=g)
    torch.cuda.synchronize()
    assert device_status() == 0
    return T_out, W, U


def full_compare(k, v, beta, C, cu, outs, io="bf16", g=None):
    T_ref, W_ref, U_ref = oracle.oracle_fwd(to64(k), to64(v), to64(beta), C, cu_seqlens=cu,
                                            g=None if g is None else to64(g))
    T_g, W_g, U_g = (to64(x) for x in outs)
    check_T(T_g, T_ref)
    check_WU(W_g, W_ref, io, "W")
    check_WU(U_g, U_ref, io, "U")
    return T_g, T_ref


# --- the specified entry point itself, kkt_solve_fwd ----------------------------------------

def _kkt_solve_fwd_call(k, v, beta, C, cu=None):
    """kkt_solve_fwd through ctypes: bf16, kernel auto, no workspace (the fixed round-robin
    schedule of the tensor-core kernel)."""
    Bt, T, H, dk = k.shape
    dv = v.shape[-1]
    T_out = torch.full((Bt, T, H, C), float("nan"), device=DEV)
    W = torch.full((Bt, T, H, dk), float("nan"), device=DEV, dtype=k.dtype)
    U = torch.full((Bt, T, H, dv), float("nan"), device=DEV, dtype=k.dtype)
    B = Bt if cu is None else cu.shape[0] - 1
    rc = _lib.lib().kkt_solve_fwd(k.data_ptr(), v.data_ptr(), beta.data_ptr(),
                                  None if cu is None else cu.data_ptr(), B, T, H, dk, dv, C,
                                  T_out.data_ptr(), W.data_ptr(), U.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.KKT_OK, _lib.status_string(rc)
    torch.cuda.synchronize()
    assert device_status() == 0
    return T_out, W, U


@pytest.mark.parametrize("C", [32, 64, 128])
@pytest.mark.parametrize("case", ["fixed", "varlen", "many_tiles"])
def test_kkt_solve_fwd_entry_point(case, C):
    """kkt_solve_fwd, the entry point with the signature the library is specified by, against the
    oracle element by element, and bit-identical to the kkt_solve_fwd_ex call with a workspace
    (the dynamic schedule that the Python front end and the bench use by default): a ragged
    fixed-length batch, a varlen batch with empty and one-token sequences, and a batch with many
    more tiles than SMs."""
    cu = None
    if case == "fixed":
        k, v, beta = make_inputs(3, 1000, 5, 128, 128, seed=101 + C, device=DEV)
    elif case == "varlen":
        lengths = [1, 63, 64, 65, 0, 130, 7, 200, 1500]
        cu = np.concatenate([[0], np.cumsum(lengths)])
        k, v, beta = make_inputs(1, int(cu[-1]), 6, 128, 128, seed=102 + C, device=DEV)
    else:
        k, v, beta = make_inputs(2, 4100, 12, 128, 128, seed=103 + C, device=DEV)
    cu_t = None if cu is None else torch.as_tensor(cu, dtype=torch.int32, device=DEV)
    outs = _kkt_solve_fwd_call(k, v, beta, C, cu_t)
    full_compare(k, v, beta, C, cu, outs)
    dyn = run(k, v, beta, C, cu, kernel="auto", workspace="auto")
    for a, b in zip(outs, dyn):
        assert torch.equal(a, b)


# --- small cases, compared in full --------------------------------------------------------

@pytest.mark.parametrize("kernel", ALL_KERNELS)
@pytest.mark.parametrize("C", [32, 64, 128])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_small_fixed_length(kernel, C, dk, dv):
    """Two sequences of 200 tokens (several chunks and a ragged tail), three heads."""
    _skip_unless(kernel, dk, dv, C)
    k, v, beta = make_inputs(2, 200, 3, dk, dv, seed=C + dk + 2 * dv, device=DEV)
    outs = run(k, v, beta, C, kernel=kernel)
    T_g, _ = full_compare(k, v, beta, C, None, outs)
    # structure: zero padding beyond the short last chunk, exact unit diagonal
    for t0, Lc in chunks(C, 2, 200):
        blk = T_g.reshape(400, 3, C)[t0:t0 + Lc]
        assert np.all(blk[:, :, Lc:] == 0.0)
        for i in range(Lc):
            assert np.all(blk[i, :, i] == 1.0) and np.all(blk[i, :, i + 1:] == 0.0)


def test_config1_fp32_io():
    """Single head, 128 tokens, C=32, dk=dv=64, fp32 in and out (SIMT kernel)."""
    w = workloads()["c1_small_f32"]
    k, v, beta, _ = w.make(seed=0, device=DEV)
    outs = run(k, v, beta, w.C)
    full_compare(k, v, beta, w.C, None, outs, io="f32")
    T = outs[0].reshape(4, 32, 32)  # the four chunks' T matrices
    assert torch.all(torch.diagonal(T, dim1=1, dim2=2) == 1.0)


@pytest.mark.parametrize("kernel", ALL_KERNELS)
@pytest.mark.parametrize("C", [32, 64, 128])
def test_small_varlen(kernel, C):
    """Packed sequences with empty, single-token, chunk-aligned and ragged lengths."""
    _skip_unless(kernel, 128, 128, C)
    lengths = [1, 63, 64, 65, 0, 130, 7, 200]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    k, v, beta = make_inputs(1, int(cu[-1]), 2, 128, 128, seed=5, device=DEV)
    outs = run(k, v, beta, C, cu, kernel=kernel)
    full_compare(k, v, beta, C, cu, outs)
    # equal to each sequence run on its own
    for s in range(len(lengths)):
        a, b = int(cu[s]), int(cu[s + 1])
        if a == b:
            continue
        alone = run(k[:, a:b].contiguous(), v[:, a:b].contiguous(), beta[:, a:b].contiguous(), C,
                    kernel=kernel)
        for x, y in zip(outs, alone):
            assert torch.equal(x[:, a:b], y)


@pytest.mark.parametrize("C", [32, 64, 128])
def test_dynamic_and_static_schedules_agree(C):
    """Tiles claimed from the workspace counter or dealt round robin: identical bits, and the
    oracle agrees (odd head count: the last head group runs past H).  A caller's workspace is
    left zero-filled by every call, so it serves the next call as it is."""
    _skip_unless("tc", 128, 128, C)
    k, v, beta = make_inputs(3, 1000, 5, 128, 128, seed=11, device=DEV)
    dyn = run(k, v, beta, C, kernel="tc", workspace="auto")
    sta = run(k, v, beta, C, kernel="tc", workspace=None)
    ws = torch.zeros(64, dtype=torch.int32, device=DEV)
    own = run(k, v, beta, C, kernel="tc", workspace=ws)
    assert torch.count_nonzero(ws).item() == 0
    again = run(k, v, beta, C, kernel="tc", workspace=ws)
    assert torch.count_nonzero(ws).item() == 0
    for a, b, c, d in zip(dyn, sta, own, again):
        assert torch.equal(a, b) and torch.equal(a, c) and torch.equal(a, d)
    full_compare(k, v, beta, C, None, dyn)


@pytest.mark.parametrize("kernel", ALL_KERNELS)
@pytest.mark.parametrize("C", [32, 64, 128])
def test_w_and_u_only_without_t(kernel, C):
    """T_out = NULL: T is computed but not written, and W, U~ are bit-identical to those of the
    materialising call (which the other tests compare with the oracle); varlen with a ragged tail."""
    _skip_unless(kernel, 128, 128, C)
    lengths = [1, 63, 64, 65, 0, 130, 7, 200]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    k, v, beta = make_inputs(1, int(cu[-1]), 3, 128, 128, seed=21, device=DEV)
    cu_t = torch.as_tensor(cu, dtype=torch.int32, device=DEV)
    T_full, W_full, U_full = run(k, v, beta, C, cu, kernel=kernel)
    W = torch.full_like(W_full, float("nan"))
    U = torch.full_like(U_full, float("nan"))
    T_none, W, U = kkt_solve_fwd(k, v, beta, C, cu_t, W_out=W, U_out=U, kernel=kernel, materialize_T=False)
    torch.cuda.synchronize()
    assert device_status() == 0
    assert T_none is None
    assert torch.equal(W, W_full) and torch.equal(U, U_full)


@pytest.mark.parametrize("kernel", ALL_KERNELS)
@pytest.mark.parametrize("C", [32, 64, 128])
@pytest.mark.parametrize("varlen", [False, True])
def test_t_out_fp16(kernel, C, varlen):
    """T_dtype = fp16: T rounded to nearest from the fp32 T, so equal to the fp32 call's T cast to
    fp16, and within 1e-4 + 2^-11 |T_ref| of the oracle (a half ulp of fp16 on top of the fp32
    bound); W, U~ bit-identical to the fp32 call's.  Fixed length with a ragged tail, or varlen."""
    _skip_unless(kernel, 128, 128, C)
    if varlen:
        lengths = [1, 63, 64, 65, 0, 130, 7, 200, 128]
        cu = np.concatenate([[0], np.cumsum(lengths)])
        k, v, beta = make_inputs(1, int(cu[-1]), 3, 128, 128, seed=23, device=DEV)
        cu_t = torch.as_tensor(cu, dtype=torch.int32, device=DEV)
    else:
        cu, cu_t = None, None
        k, v, beta = make_inputs(2, 3 * C + 17, 5, 128, 128, seed=24, device=DEV)
    T32, W32, U32 = run(k, v, beta, C, cu, kernel=kernel)
    T16 = torch.full(T32.shape, float("nan"), device=DEV, dtype=torch.float16)
    W = torch.full_like(W32, float("nan"))
    U = torch.full_like(U32, float("nan"))
    kkt_solve_fwd(k, v, beta, C, cu_t, T_out=T16, W_out=W, U_out=U, kernel=kernel, T_dtype=torch.float16)
    torch.cuda.synchronize()
    assert device_status() == 0
    assert torch.equal(T16, T32.to(torch.float16))
    assert torch.equal(W, W32) and torch.equal(U, U32)
    T_ref, _, _ = oracle.oracle_fwd(to64(k), to64(v), to64(beta), C, cu_seqlens=cu)
    err = np.abs(to64(T16) - T_ref)
    assert (err <= 1e-4 + 2.0 ** -11 * np.abs(T_ref)).all(), float(err.max())


# --- the gated variant (diag(beta)(Gamma o K K^T)) --------------------------------------------

@pytest.mark.parametrize("kernel", ALL_KERNELS)
@pytest.mark.parametrize("C", [32, 64, 128])
@pytest.mark.parametrize("varlen", [False, True])
def test_gated(kernel, C, varlen):
    """Gated coefficient against the oracle, element by element: fixed length with a ragged tail and
    a partial head group, or varlen with empty and one-token sequences."""
    _skip_unless(kernel, 128, 128, C)
    if varlen:
        lengths = [1, 63, 64, 65, 0, 130, 7, 200, 128]
        cu = np.concatenate([[0], np.cumsum(lengths)])
        k, v, beta = make_inputs(1, int(cu[-1]), 3, 128, 128, seed=41, device=DEV)
        g = make_gate(1, int(cu[-1]), 3, seed=41, device=DEV)
    else:
        cu = None
        k, v, beta = make_inputs(2, 3 * C + 17, 5, 128, 128, seed=42, device=DEV)
        g = make_gate(2, 3 * C + 17, 5, seed=42, device=DEV)
    outs = run(k, v, beta, C, cu, kernel=kernel, g=g)
    full_compare(k, v, beta, C, cu, outs, g=g)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128)])
def test_gated_simt_shapes_and_fp32(dk, dv):
    """The SIMT kernel's gated path at d = 64 and with fp32 I/O (the fp32 workload's shapes)."""
    k, v, beta = make_inputs(1, 200, 2, dk, dv, seed=43, device=DEV)
    g = make_gate(1, 200, 2, seed=43, device=DEV)
    full_compare(k, v, beta, 64, None, run(k, v, beta, 64, kernel="simt", g=g), g=g)
    kf, vf, bf = make_inputs(1, 128, 1, dk, dv, seed=44, dtype=torch.float32, device=DEV)
    gf = make_gate(1, 128, 1, seed=44, device=DEV)
    full_compare(kf, vf, bf, 32, None, run(kf, vf, bf, 32, kernel="simt", g=gf), io="f32", g=gf)


@pytest.mark.parametrize("kernel", ALL_KERNELS)
def test_gate_zero_is_ungated(kernel):
    """g = 0 (no decay): the gated call returns exactly the ungated call's T, W and U~."""
    _skip_unless(kernel, 128, 128, 64)
    k, v, beta = make_inputs(2, 300, 4, 128, 128, seed=45, device=DEV)
    plain = run(k, v, beta, 64, kernel=kernel)
    gated = run(k, v, beta, 64, kernel=kernel, g=torch.zeros_like(beta))
    for a, b in zip(plain, gated):
        assert torch.equal(a, b)


@pytest.mark.parametrize("kernel", ALL_KERNELS)
@pytest.mark.parametrize("C", [32, 64, 128])
def test_gate_cut_is_block_diagonal(kernel, C):
    """A token with zero decay (g = -1000) cuts its chunk: T is exactly zero across the cut, and the
    rest matches the oracle.  The cuts make their blocks of the decay matrix non-factorable, so the
    element-by-element path runs (at C = 128 also where M10 of the level-64 coupling is formed)."""
    _skip_unless(kernel, 128, 128, C)
    k, v, beta = make_inputs(1, 256, 2, 128, 128, seed=46, device=DEV)
    g = make_gate(1, 256, 2, seed=46, device=DEV)
    cuts = {32: [(10, 0), (32 + 20, 1), (128 + 5, 0)],
            64: [(40, 0), (64 + 33, 1), (128 + 64 + 5, 0)],
            128: [(40, 0), (100, 1), (128 + 70, 0)]}[C]
    for t, h in cuts:
        g[0, t, h] = -1000.0
    T, W, U = run(k, v, beta, C, kernel=kernel, g=g)
    for t, h in cuts:
        c0, cut = (t // C) * C, t % C
        blk = T[0, c0 + cut:c0 + C, h, :cut]
        assert torch.count_nonzero(blk) == 0
    full_compare(k, v, beta, C, None, (T, W, U), g=g)


@pytest.mark.parametrize("C", [32, 64, 128])
@pytest.mark.parametrize("variant", ["plain", "gated", "t_fp16", "no_t"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (64, 128)])
def test_tc_head_dims(C, variant, dk, dv):
    """The tensor-core kernel at the head dimensions other than 128 / 128: d_k = d_v = 64 (one
    64-column box per row, N = 128 for W|U~) and the mixed pairs (N = 192): varlen with empty and
    one-token sequences and a ragged tail, every variant, against the oracle (W and U~ only:
    bit-identical to the materialising call)."""
    lengths = [1, 63, 64, 65, 0, 130, 7, 200, 128]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    k, v, beta = make_inputs(1, int(cu[-1]), 3, dk, dv, seed=C + 91, device=DEV)
    g = make_gate(1, int(cu[-1]), 3, seed=C + 91, device=DEV) if variant == "gated" else None
    assert select_kernel(dk, dv, C) == "tc"
    outs = run(k, v, beta, C, cu, kernel="tc", g=g)
    full_compare(k, v, beta, C, cu, outs, g=g)
    cu_t = torch.as_tensor(cu, dtype=torch.int32, device=DEV)
    if variant == "t_fp16":
        T16, W, U = kkt_solve_fwd(k, v, beta, C, cu_t, kernel="tc", T_dtype=torch.float16)
        torch.cuda.synchronize()
        assert torch.equal(T16, outs[0].to(torch.float16))
        assert torch.equal(W, outs[1]) and torch.equal(U, outs[2])
    if variant == "no_t":
        T_none, W, U = kkt_solve_fwd(k, v, beta, C, cu_t, kernel="tc", materialize_T=False)
        torch.cuda.synchronize()
        assert T_none is None and torch.equal(W, outs[1]) and torch.equal(U, outs[2])


# --- degenerate cases and traps -----------------------------------------------------------

@pytest.mark.parametrize("kernel", ALL_KERNELS)
def test_beta_zero_gives_identity(kernel):
    """beta = 0: T = I exactly, W = U = 0 (degenerate test 1 of the page's section 4)."""
    _skip_unless(kernel, 128, 128, 64)
    k, v, beta = make_inputs(1, 256, 2, 128, 128, seed=3, device=DEV)
    T, W, U = run(k, v, torch.zeros_like(beta), 64, kernel=kernel)
    eye = torch.eye(64, device=DEV).repeat(4, 1).reshape(256, 1, 64).expand(256, 2, 64)
    assert torch.equal(T[0], eye)
    assert torch.all(W == 0) and torch.all(U == 0)


@pytest.mark.parametrize("kernel", ALL_KERNELS)
def test_subdiagonal_block_sign(kernel):
    """Only L10 nonzero (L00 = L11 = I): T's lower-left block is -L10 (degenerate test 2)."""
    _skip_unless(kernel, 128, 128, 32)
    rng = np.random.default_rng(4)
    beta = rng.integers(1, 64, 32) / 64.0
    kk, L10 = subdiagonal_only_case(beta)
    k = torch.zeros((1, 32, 1, 128), dtype=torch.bfloat16)
    k[0, :, 0, :32] = torch.from_numpy(kk).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((1, 32, 1, 128))).to(torch.bfloat16)
    b = torch.from_numpy(beta).float().reshape(1, 32, 1)
    T, W, U = run(k.to(DEV), v.to(DEV), b.to(DEV), 32, kernel=kernel)
    Tn = to64(T)[0, :, 0, :]
    np.testing.assert_allclose(Tn[16:, :16], -L10, atol=1e-6, rtol=0)
    np.testing.assert_array_equal(Tn[:16, :16], np.eye(16))
    np.testing.assert_array_equal(Tn[16:, 16:], np.eye(16))


@pytest.mark.parametrize("kernel", ALL_KERNELS)
def test_no_state_carried_between_chunks(kernel):
    """Chunks with beta = 0 between ordinary ones stay exactly the identity, so no buffer
    reused across chunks leaks the previous chunk's values (section 3.6 trap)."""
    _skip_unless(kernel, 128, 128, 64)
    k, v, beta = make_inputs(2, 64 * 40, 4, 128, 128, seed=9, device=DEV)
    mask = torch.zeros(2, 40, 1, 4, device=DEV)
    mask[:, 1::3] = 1.0
    beta0 = (beta.reshape(2, 40, 64, 4) * (1 - mask)).reshape_as(beta).contiguous()
    T, W, U = run(k, v, beta0, 64, kernel=kernel)
    Tz = T.reshape(2, 40, 64, 4, 64)[:, 1::3]
    eye = torch.eye(64, device=DEV).reshape(1, 1, 64, 1, 64)
    assert torch.equal(Tz, eye.expand_as(Tz))
    assert torch.all(W.reshape(2, 40, 64, 4, 128)[:, 1::3] == 0)
    full_compare(k, v, beta0, 64, None, (T, W, U))


def test_malformed_cu_seqlens_is_reported_not_faulted():
    """A decreasing cu_seqlens is skipped by the kernel and reported by the status word."""
    k, v, beta = make_inputs(1, 300, 2, 128, 128, seed=6, device=DEV)
    cu = torch.tensor([0, 200, 100, 300], dtype=torch.int32, device=DEV)
    T_out = torch.zeros((1, 300, 2, 64), device=DEV)
    W = torch.zeros((1, 300, 2, 128), device=DEV, dtype=torch.bfloat16)
    U = torch.zeros_like(W)
    kkt_solve_fwd(k, v, beta, 64, cu, T_out=T_out, W_out=W, U_out=U)
    assert device_status() == _lib.KKT_ERR_SEQLENS
    assert device_status() == 0
    cu_ok = np.array([0, 100, 300])
    outs = run(k, v, beta, 64, cu_ok)
    full_compare(k, v, beta, 64, cu_ok, outs)


def test_checked_mode_raises_device_errors(monkeypatch):
    """check=True (or KKT_CHECK=1) reads the status word after the call and raises on a device error."""
    k, v, beta = make_inputs(1, 300, 2, 128, 128, seed=6, device=DEV)
    bad = torch.tensor([0, 200, 100, 300], dtype=torch.int32, device=DEV)
    with pytest.raises(_lib.KktError) as e:
        kkt_solve_fwd(k, v, beta, 64, bad, check=True)
    assert e.value.status == _lib.KKT_ERR_SEQLENS
    monkeypatch.setenv("KKT_CHECK", "1")
    with pytest.raises(_lib.KktError):
        kkt_solve_fwd(k, v, beta, 64, bad)
    good = torch.tensor([0, 100, 300], dtype=torch.int32, device=DEV)
    kkt_solve_fwd(k, v, beta, 64, good)  # checked, no error
    assert device_status() == 0


# (full-size workloads: every element, tests/test_full_size_gpu.py)


@pytest.mark.parametrize("kernel", ALL_KERNELS)
def test_cuda_graph_capture_and_replay(kernel):
    """Calls captured into a CUDA graph replay to the eager results, bit for bit: the launch carries
    no host state between calls (the work counter in the workspace clears itself), so replays
    and back-to-back launches with programmatic dependent launch are safe."""
    _skip_unless(kernel, 128, 128, 64)
    k, v, beta = make_inputs(2, 700, 3, 128, 128, seed=51, device=DEV)
    g = make_gate(2, 700, 3, seed=51, device=DEV)
    eager = run(k, v, beta, 64, kernel=kernel)
    eager_g = run(k, v, beta, 64, kernel=kernel, g=g)
    T1, W1, U1 = (torch.full_like(x, float("nan")) for x in eager)
    T2, W2, U2 = (torch.full_like(x, float("nan")) for x in eager_g)
    ws = torch.zeros(64, dtype=torch.int32, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up on the capture stream
        kkt_solve_fwd(k, v, beta, 64, T_out=T1, W_out=W1, U_out=U1, kernel=kernel, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(3):
            kkt_solve_fwd(k, v, beta, 64, T_out=T1, W_out=W1, U_out=U1, kernel=kernel, workspace=ws)
            kkt_solve_fwd(k, v, beta, 64, T_out=T2, W_out=W2, U_out=U2, kernel=kernel, workspace=ws, g=g)
    for x in (T1, W1, U1, T2, W2, U2):
        x.fill_(float("nan"))
    for _ in range(4):
        graph.replay()
    torch.cuda.synchronize()
    assert device_status() == 0
    assert torch.count_nonzero(ws).item() == 0
    for a, b in zip(eager + eager_g, (T1, W1, U1, T2, W2, U2)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("case", ["batch", "one_long_sequence", "varlen", "gated_fp16"])
def test_host_runner_pipeline(case):
    """The end-to-end runner (pinned host buffers, the batch cut into pieces that are copied in,
    solved and copied out on overlapping streams) returns exactly what one device call returns."""
    from gdn_chunkwise_ut_gb300 import HostRunner
    C, H = 64, 3
    cu, g, t_dtype = None, None, torch.float32
    if case == "batch":
        k, v, beta = make_inputs(4, 700, H, 128, 128, seed=81, device=DEV)
    elif case == "one_long_sequence":
        k, v, beta = make_inputs(1, 3000, H, 128, 128, seed=82, device=DEV)
    else:
        lengths = [1, 63, 64, 0, 700, 130, 7, 1200, 5]
        cu = np.concatenate([[0], np.cumsum(lengths)])
        k, v, beta = make_inputs(1, int(cu[-1]), H, 128, 128, seed=83, device=DEV)
        if case == "gated_fp16":
            g = make_gate(1, int(cu[-1]), H, seed=83, device=DEV)
            t_dtype = torch.float16
    cu_t = None if cu is None else torch.as_tensor(cu, dtype=torch.int32, device=DEV)
    ref = kkt_solve_fwd(k, v, beta, C, cu_t, g=g, T_dtype=t_dtype)
    torch.cuda.synchronize()
    runner = HostRunner(k.shape[0], k.shape[1], H, 128, 128, C, cu_seqlens=cu, T_dtype=t_dtype,
                        gated=g is not None, pieces=4)
    hosts = [x.cpu().pin_memory() for x in (k, v, beta)]
    gh = g.cpu().pin_memory() if g is not None else None
    for _ in range(2):  # a second call reuses the buffers
        outs = runner(*hosts, g_host=gh)
        for a, b in zip(ref, outs):
            assert torch.equal(a.cpu(), b)
    assert device_status() == 0
