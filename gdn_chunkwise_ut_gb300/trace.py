"""Pipeline trace of the tensor-core kernel (a profiling aid, not part of the product path).

Builds libkkt_trace.so (the same sources compiled with -DKKT_TRACE), runs one
workload and prints, for the first CTAs, when each role reached each event of
every tile (microseconds from the CTA's first event), plus per-role averages:

    python -m gdn_chunkwise_ut_gb300.trace [--workload c3_b4_t8192_h16] [--ctas 2] [--tiles 12]
"""
from __future__ import annotations

import argparse
import ctypes

import numpy as np
import torch

from . import _lib, build
from .inputs import workloads

EVENTS = ["P_EMPTY", "P_ISSUE", "M_FULL", "M_GRAM", "M_EPI", "I_GRAM", "I_INV", "I_TSTORE", "I_TT",
          "E_DFULL", "E_DEMPTY", "E_DONE", "I_LD", "I_DIAG", "I_C16", "I_PAIR"]
TRACE_CTAS, TRACE_TILES, TRACE_SLOTS = 160, 64, 16


def run(workload: str, warmup: int = 3, dynamic: bool = True):
    path = build.build(trace=True)
    lib = _lib.lib(path)
    lib.kkt_set_trace_buffer.argtypes = [ctypes.c_void_p]
    lib.kkt_set_trace_buffer.restype = None
    w = workloads()[workload]
    k, v, beta, cu = w.make(seed=0, device="cuda")
    cu_t = None if cu is None else torch.as_tensor(cu, dtype=torch.int32, device="cuda")
    B = len(cu) - 1 if cu is not None else w.B
    T_out = torch.empty((k.shape[0], k.shape[1], w.H, w.C), device="cuda")
    W = torch.empty_like(k)
    U = torch.empty_like(v)
    buf = torch.zeros(TRACE_CTAS * TRACE_TILES * TRACE_SLOTS, dtype=torch.int64, device="cuda")
    ws = torch.zeros(_lib.KKT_WORKSPACE_BYTES // 4, dtype=torch.int32, device="cuda") if dynamic else None
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        rc = lib.kkt_solve_fwd_ex(k.data_ptr(), v.data_ptr(), beta.data_ptr(),
                                  None if cu_t is None else cu_t.data_ptr(), B, k.shape[1], w.H, w.dk, w.dv,
                                  w.C, T_out.data_ptr(), W.data_ptr(), U.data_ptr(), _lib.KKT_IO_BF16,
                                  _lib.KKT_KERNEL_TC, None if ws is None else ws.data_ptr(),
                                  0 if ws is None else ws.numel() * 4, stream)
        if rc != 0:
            raise _lib.KktError(rc, "kkt_solve_fwd_ex")

    for _ in range(warmup):
        call()
    lib.kkt_set_trace_buffer(buf.data_ptr())
    call()
    torch.cuda.synchronize()
    lib.kkt_set_trace_buffer(None)
    return buf.cpu().numpy().reshape(TRACE_CTAS, TRACE_TILES, TRACE_SLOTS)[:, :, :len(EVENTS)]


def report(tr: np.ndarray, ctas: int, tiles: int) -> str:
    lines = []
    for b in range(ctas):
        t = tr[b].astype(np.float64)
        valid = t > 0
        if not valid.any():
            continue
        t0 = t[valid].min()
        us = np.where(valid, (t - t0) / 1e3, np.nan)
        lines.append(f"CTA {b} (us from its first event)")
        lines.append("tile " + " ".join(f"{e:>9s}" for e in EVENTS[:12]))
        for i in range(min(tiles, us.shape[0])):
            if not np.isfinite(us[i]).any():
                break
            lines.append(f"{i:4d} " + " ".join(f"{x:9.2f}" if np.isfinite(x) else f"{'':9s}" for x in us[i][:12]))
    # averages over all traced CTAs and tiles (steady state: skip the first two tiles)
    t = tr.astype(np.float64)
    ev = {e: i for i, e in enumerate(EVENTS)}

    def span(a, b_):
        x = t[:, 2:, ev[b_]] - t[:, 2:, ev[a]]
        ok = (t[:, 2:, ev[a]] > 0) & (t[:, 2:, ev[b_]] > 0)
        return float(np.mean(x[ok])) / 1e3 if ok.any() else float("nan")

    def period(e):
        x = np.diff(t[:, :, ev[e]], axis=1)
        ok = (t[:, 1:, ev[e]] > 0) & (t[:, :-1, ev[e]] > 0)
        return float(np.mean(x[:, 1:][ok[:, 1:]])) / 1e3 if ok[:, 1:].any() else float("nan")

    # whole grid: first event and last epilogue completion per CTA
    starts, ends, ntiles = [], [], []
    for b in range(t.shape[0]):
        tb = t[b]
        if not (tb > 0).any():
            continue
        starts.append(tb[tb > 0].min())
        done = tb[:, ev["E_DONE"]]
        ends.append(done[done > 0].max() if (done > 0).any() else np.nan)
        ntiles.append(int((done > 0).sum()))
    if starts:
        g0 = min(starts)
        st = (np.array(starts) - g0) / 1e3
        en = (np.array(ends) - g0) / 1e3
        nt = np.array(ntiles)
        lines.append("")
        lines.append(f"grid: {len(st)} CTAs traced; start spread {st.min():.2f}..{st.max():.2f} us; "
                     f"end {np.nanmin(en):.2f}..{np.nanmax(en):.2f} us (median {np.nanmedian(en):.2f}); "
                     f"tiles per CTA {nt.min()}..{nt.max()}")
        for k_ in sorted(set(nt.tolist())):
            sel = nt == k_
            lines.append(f"  CTAs with {k_} tiles: {sel.sum()}, end {np.nanmin(en[sel]):.2f}..{np.nanmax(en[sel]):.2f} us")
    lines.append("")
    lines.append(f"period per tile (M_EPI to M_EPI)         {period('M_EPI'):7.2f} us")
    lines.append(f"load: issue -> landed (P_ISSUE->M_FULL)  {span('P_ISSUE', 'M_FULL'):7.2f} us")
    lines.append(f"inverse: Gram ready -> T~ written        {span('I_GRAM', 'I_TT'):7.2f} us")
    lines.append(f"  Gram row load + L row                  {span('I_GRAM', 'I_LD'):7.2f} us")
    lines.append(f"  16x16 diagonal substitution            {span('I_LD', 'I_DIAG'):7.2f} us")
    lines.append(f"  level-16 coupling                      {span('I_DIAG', 'I_C16'):7.2f} us")
    lines.append(f"  pair sync                              {span('I_C16', 'I_PAIR'):7.2f} us")
    lines.append(f"  level-32 coupling                      {span('I_PAIR', 'I_INV'):7.2f} us")
    lines.append(f"  T store                                {span('I_INV', 'I_TSTORE'):7.2f} us")
    lines.append(f"  wait T~ free + write T~                {span('I_TSTORE', 'I_TT'):7.2f} us")
    lines.append(f"Gram issued -> inverse starts            {span('M_GRAM', 'I_GRAM'):7.2f} us")
    lines.append(f"T~ written -> W|U MMA issued             {span('I_TT', 'M_EPI'):7.2f} us")
    lines.append(f"W|U MMA issued -> epilogue starts        {span('M_EPI', 'E_DFULL'):7.2f} us")
    lines.append(f"epilogue: D loads                        {span('E_DFULL', 'E_DEMPTY'):7.2f} us")
    lines.append(f"epilogue: total                          {span('E_DFULL', 'E_DONE'):7.2f} us")
    lines.append(f"stage empty wait -> issue                {span('P_EMPTY', 'P_ISSUE'):7.2f} us")
    return "\n".join(lines)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="c3_b4_t8192_h16")
    ap.add_argument("--ctas", type=int, default=2)
    ap.add_argument("--tiles", type=int, default=12)
    ap.add_argument("--static", action="store_true", help="fixed round-robin schedule (no workspace)")
    a = ap.parse_args()
    print(report(run(a.workload, dynamic=not a.static), a.ctas, a.tiles))


if __name__ == "__main__":
    main()
