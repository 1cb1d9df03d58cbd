"""Runs one workload a few times through the C ABI, for profilers (ncu) to capture.

    python -m gdn_chunkwise_ut_gb300.profile_case [--workload c3_b4_t8192_h16] [--calls 4] [--kernel auto]
        [--gated] [--consumer] [--head-dim 64]

``--consumer`` runs the chunk state recurrence (gdn_chunk_state_fwd) ``--calls`` times instead, on W and
U~ from one kkt_solve call.

No timing and no checking: inputs are generated once, then ``--calls`` launches
of the path run back to back and the process synchronises and exits.
"""
from __future__ import annotations

import argparse
import dataclasses

import torch

from .api import gdn_chunk_state_fwd, kkt_solve_fwd
from .inputs import make_gate, make_query, make_state, workloads


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="c3_b4_t8192_h16")
    ap.add_argument("--calls", type=int, default=4)
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "tc"])
    ap.add_argument("--gated", action="store_true", help="the gated variant (seeded log decays)")
    ap.add_argument("--consumer", action="store_true", help="the chunk state recurrence instead of kkt_solve")
    ap.add_argument("--head-dim", type=int, default=None, help="override d_k = d_v (64 or 128)")
    a = ap.parse_args()
    w = workloads()[a.workload]
    if a.head_dim is not None:
        w = dataclasses.replace(w, dk=a.head_dim, dv=a.head_dim)
    k, v, beta, cu = w.make(seed=0, device="cuda")
    g = make_gate(k.shape[0], k.shape[1], w.H, device="cuda") if a.gated else None
    cu_t = None if cu is None else torch.as_tensor(cu, dtype=torch.int32, device="cuda")
    if a.consumer:
        q = make_query(k.shape[0], k.shape[1], w.H, w.dk, device="cuda")
        N = w.B if cu is None else len(cu) - 1
        S0 = make_state(N, w.H, w.dk, w.dv, device="cuda")
        _, W, U = kkt_solve_fwd(k, v, beta, w.C, cu_t, materialize_T=False, g=g)
        o = S = None
        for _ in range(a.calls):
            o, S = gdn_chunk_state_fwd(q, k, W, U, w.C, g=g, initial_state=S0, cu_seqlens=cu_t, o=o, final_state=S)
        torch.cuda.synchronize()
        print(f"{a.calls} recurrence calls of {a.workload}{' (gated)' if a.gated else ''}")
        return
    outs = None
    for _ in range(a.calls):
        outs = kkt_solve_fwd(k, v, beta, w.C, cu_t, kernel=a.kernel,
                             T_out=None if outs is None else outs[0],
                             W_out=None if outs is None else outs[1],
                             U_out=None if outs is None else outs[2], g=g)
    torch.cuda.synchronize()
    print(f"{a.calls} calls of {a.workload} ({a.kernel}{', gated' if a.gated else ''})")


if __name__ == "__main__":
    main()
