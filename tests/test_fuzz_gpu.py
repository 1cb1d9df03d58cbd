"""Seeded random shapes against the fp64 oracle (GPU).

Each case draws a chunk size, head dimensions (equal or not, so both kernels run), a head count,
fixed-length or packed variable-length sequences (empty and one-token ones included), and a
variant (plain, gated, fp16 T, W and U~ only), and compares the whole output with the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from gdn_chunkwise_ut_gb300 import device_status, kkt_solve_fwd, select_kernel
from gdn_chunkwise_ut_gb300.inputs import make_gate, make_inputs
from tests.compare import check_T, check_WU, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    C = int(rng.choice([32, 64, 128]))
    dk = int(rng.choice([64, 128]))
    dv = dk if rng.random() < 0.7 else int(rng.choice([64, 128]))
    H = int(rng.integers(1, 7))
    if rng.random() < 0.5:
        lengths = rng.integers(0, 330, int(rng.integers(1, 7)))
        lengths[rng.random(len(lengths)) < 0.2] = int(rng.choice([0, 1]))
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
        B, T = 1, int(cu[-1])
    else:
        cu, B, T = None, int(rng.integers(1, 4)), int(rng.integers(1, 330))
    variant = str(rng.choice(["plain", "gated", "t_fp16", "no_t"]))
    return C, dk, dv, H, B, T, cu, variant


@pytest.mark.parametrize("seed", range(24))
def test_random_shapes(seed):
    C, dk, dv, H, B, T, cu, variant = _case(seed)
    if T == 0:
        pytest.skip("no tokens")
    k, v, beta = make_inputs(B, T, H, dk, dv, seed=seed, device=DEV)
    g = make_gate(B, T, H, seed=seed, device=DEV) if variant == "gated" else None
    cu_t = None if cu is None else torch.as_tensor(cu, dtype=torch.int32, device=DEV)
    t_dtype = torch.float16 if variant == "t_fp16" else torch.float32
    T_out, W, U = kkt_solve_fwd(k, v, beta, C, cu_t, g=g, T_dtype=t_dtype, materialize_T=variant != "no_t",
                                check=True)
    torch.cuda.synchronize()
    assert device_status() == 0
    T_ref, W_ref, U_ref = oracle.oracle_fwd(to64(k), to64(v), to64(beta), C, cu_seqlens=cu,
                                            g=None if g is None else to64(g))
    what = f"C={C} dk={dk} dv={dv} H={H} B={B} T={T} varlen={cu is not None} {variant} " \
           f"kernel={select_kernel(dk, dv, C)}"
    if T_out is not None:
        T_g = to64(T_out)
        if variant == "t_fp16":
            assert (np.abs(T_g - T_ref) <= 1e-4 + 2.0 ** -11 * np.abs(T_ref)).all(), what
        else:
            check_T(T_g, T_ref, what)
    check_WU(to64(W), W_ref, "bf16", "W " + what)
    check_WU(to64(U), U_ref, "bf16", "U " + what)
