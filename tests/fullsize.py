"""Whole-tensor oracle parity of a full-size workload, in the bench's launch configuration.

Shared by ``tests/test_full_size_gpu.py`` (the assertions) and ``tests/parity_report.py`` (the
table of errors per workload).  The library runs the whole workload in one call (kernel "auto",
the cached workspace: what ``bench.py`` times); the oracle then runs slab by slab (groups of whole
sequences) on the same bf16-rounded inputs, and every element of T, W and U~ is compared.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gdn_chunkwise_ut_gb300 import device_status, kkt_solve_fwd
from gdn_chunkwise_ut_gb300.inputs import make_gate, workloads
from tests.compare import FullComparison, chunks, slabs, to64

PLAIN = ["c1_small_f32", "c2_t8192_h16"] + [f"c3_b4_t8192_h{H}" for H in (64, 48, 32, 24, 16, 8)] + \
        ["c4_varlen32_h32"] + [f"c5_b2_t16384_h24_c{C}" for C in (32, 64, 128)]
GATED = ["c2_t8192_h16", "c3_b4_t8192_h16", "c4_varlen32_h32"] + \
        [f"c5_b2_t16384_h24_c{C}" for C in (32, 64, 128)]


def run_and_compare(name: str, gated: bool = False, seed: int = 0, device: str = "cuda") -> dict:
    w = workloads()[name]
    k, v, beta, cu = w.make(seed=seed, device=device)
    g = make_gate(k.shape[0], k.shape[1], w.H, seed=seed, device=device) if gated else None
    cu_t = None if cu is None else torch.as_tensor(cu, dtype=torch.int32, device=device)
    T_out = torch.full((k.shape[0], k.shape[1], w.H, w.C), float("nan"), device=device)
    W = torch.full(k.shape, float("nan"), device=device, dtype=k.dtype)
    U = torch.full(v.shape, float("nan"), device=device, dtype=v.dtype)
    kkt_solve_fwd(k, v, beta, w.C, cu_t, T_out=T_out, W_out=W, U_out=U, g=g)
    torch.cuda.synchronize()
    assert device_status() == 0
    H, C, N = w.H, w.C, w.tokens
    flat = lambda x: x.reshape(N, H, -1)
    kf, vf, bf = flat(k), flat(v), beta.reshape(N, H)
    gf = None if g is None else g.reshape(N, H)
    Tf, Wf, Uf = flat(T_out), flat(W), flat(U)

    # structure over the whole tensor: unit diagonal and zero upper triangle of every chunk
    starts = torch.zeros(N, dtype=torch.long, device=device)
    for t0, Lc in chunks(C, w.B, w.T, cu):
        starts[t0:t0 + Lc] = t0
    row = (torch.arange(N, device=device) - starts).reshape(-1, 1, 1)
    col = torch.arange(C, device=device).reshape(1, 1, C)
    assert torch.all(Tf[(col == row).expand_as(Tf)] == 1.0)
    assert torch.all(Tf[(col > row).expand_as(Tf)] == 0.0)

    acc = FullComparison(w.io)
    nthreads = 0  # every host core
    for n0, n1, cu_rel in slabs(w.B, w.T, cu, max_tokens=max(1, (1 << 19) // H)):
        n = n1 - n0
        if cu_rel is None:
            nb = n // w.T
            shape = lambda x, d: to64(x[n0:n1]).reshape(nb, w.T, H, d) if d else to64(x[n0:n1]).reshape(nb, w.T, H)
        else:
            shape = lambda x, d: to64(x[n0:n1]).reshape(1, n, H, d) if d else to64(x[n0:n1]).reshape(1, n, H)
        T_ref, W_ref, U_ref = oracle.oracle_fwd(shape(kf, w.dk), shape(vf, w.dv), shape(bf, 0), C,
                                                cu_seqlens=cu_rel, nthreads=nthreads,
                                                g=None if gf is None else shape(gf, 0))
        acc.add(to64(Tf[n0:n1]).reshape(T_ref.shape), to64(Wf[n0:n1]).reshape(W_ref.shape),
                to64(Uf[n0:n1]).reshape(U_ref.shape), T_ref, W_ref, U_ref)
    out = acc.finish()
    out.update(name=name, gated=gated, tokens=N, heads=H, C=C)
    return out
