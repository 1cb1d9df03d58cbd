"""Pipeline trace of the tensor-core kernel (a profiling aid, not part of the product path).

Builds libkkt_trace.so (the same sources compiled with -DKKT_TRACE), runs one
workload and prints, for the first CTAs, when each role reached each event of
every tile (microseconds from the CTA's first event), plus per-role averages.
Events are SM cycle counts, mapped to the global timer with the pairs of
(global timer, cycle count) that each CTA records at its start and end.

    python -m gdn_chunkwise_ut_gb300.trace [--workload c3_b4_t8192_h16] [--ctas 2] [--tiles 12] [--head-dim 64]
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses

import numpy as np
import torch

from . import _lib, build
from .inputs import make_gate, workloads

EVENTS = ["P_EMPTY", "P_ISSUE", "M_FULL", "M_GRAM", "M_EPI", "I_GRAM", "I_INV", "I_TSTORE", "I_TT",
          "E_DFULL", "E_DEMPTY", "E_DONE", "I_LD", "I_DIAG", "I_C16", "I_PAIR", "M_LATE", "M_READY", "I_BW", "I_TTW",
          "I_L32", "I_L32B", "I_M11", "I_Y", "I_YB", "I_Z", "I_INVB", "I_OPS", "E_M10", "M_L64Y", "M_L64Z",
          "I_SPLIT", "I_YSPL"]
TRACE_CTAS, TRACE_TILES, TRACE_SLOTS = 160, 64, 40


def run(workload: str, warmup: int = 3, dynamic: bool = True, gated: bool = False, head_dim: int | None = None):
    path = build.build(trace=True)
    lib = _lib.lib(path)
    lib.kkt_set_trace_buffer.argtypes = [ctypes.c_void_p]
    lib.kkt_set_trace_buffer.restype = None
    w = workloads()[workload]
    if head_dim is not None:
        w = dataclasses.replace(w, dk=head_dim, dv=head_dim)
    k, v, beta, cu = w.make(seed=0, device="cuda")
    cu_t = None if cu is None else torch.as_tensor(cu, dtype=torch.int32, device="cuda")
    B = len(cu) - 1 if cu is not None else w.B
    g = make_gate(k.shape[0], k.shape[1], w.H, device="cuda") if gated else None
    T_out = torch.empty((k.shape[0], k.shape[1], w.H, w.C), device="cuda")
    W = torch.empty_like(k)
    U = torch.empty_like(v)
    buf = torch.zeros(TRACE_CTAS * TRACE_TILES * TRACE_SLOTS, dtype=torch.int64, device="cuda")
    ws = torch.zeros(_lib.KKT_WORKSPACE_BYTES // 4, dtype=torch.int32, device="cuda") if dynamic else None
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        rc = lib.kkt_solve_fwd_gated(k.data_ptr(), v.data_ptr(), beta.data_ptr(),
                                     None if g is None else g.data_ptr(),
                                     None if cu_t is None else cu_t.data_ptr(), B, k.shape[1], w.H, w.dk, w.dv,
                                     w.C, T_out.data_ptr(), W.data_ptr(), U.data_ptr(), _lib.KKT_IO_BF16,
                                     _lib.KKT_KERNEL_TC, None if ws is None else ws.data_ptr(),
                                     0 if ws is None else ws.numel() * 4, stream)
        if rc != 0:
            raise _lib.KktError(rc, "kkt_solve_fwd_ex")

    for _ in range(warmup):
        call()
    # untraced launches of the trace build, timed with CUDA events on the launching stream
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    torch.cuda.synchronize()
    ev0.record()
    for _ in range(reps):
        call()
    ev1.record()
    torch.cuda.synchronize()
    run.last_ms = ev0.elapsed_time(ev1) / reps
    lib.kkt_set_trace_buffer(buf.data_ptr())
    call()
    torch.cuda.synchronize()
    lib.kkt_set_trace_buffer(None)
    raw = buf.cpu().numpy().reshape(TRACE_CTAS, TRACE_TILES, TRACE_SLOTS)
    run.last_raw = raw
    return to_ns(raw)


def to_ns(raw: np.ndarray) -> np.ndarray:
    """Cycle counts -> global-timer ns per CTA (NaN where an event was not recorded)."""
    cal = raw[:, -1, :4].astype(np.float64)  # g0, c0, g1, c1
    ev = raw[:, :-1, :len(EVENTS)].astype(np.float64)
    out = np.full(ev.shape, np.nan)
    for b in range(raw.shape[0]):
        g0, c0, g1, c1 = cal[b]
        if c1 <= c0 or g1 <= g0:
            continue
        ns_per_clk = (g1 - g0) / (c1 - c0)
        ok = ev[b] > 0
        out[b][ok] = g0 + (ev[b][ok] - c0) * ns_per_clk
    return out


def report(tr: np.ndarray, ctas: int, tiles: int) -> str:
    lines = []
    shown = EVENTS[:12] + ["M_LATE", "M_READY"]
    idx = [EVENTS.index(e) for e in shown]
    for b in range(ctas):
        t = tr[b]
        if not np.isfinite(t).any():
            continue
        us = (t - np.nanmin(t)) / 1e3
        lines.append(f"CTA {b} (us from its first event)")
        lines.append("tile " + " ".join(f"{e:>9s}" for e in shown))
        for i in range(min(tiles, us.shape[0])):
            if not np.isfinite(us[i]).any():
                break
            lines.append(f"{i:4d} " + " ".join(f"{us[i][k]:9.2f}" if np.isfinite(us[i][k]) else f"{'':9s}" for k in idx))
    # averages over all traced CTAs and tiles (steady state: skip the first two tiles)
    t = tr
    ev = {e: i for i, e in enumerate(EVENTS)}

    def span(a, b_, shift=0):
        """mean of event b_ of tile i + shift minus event a of tile i"""
        x = t[:, 2:t.shape[1] - shift, ev[b_]] if shift == 0 else t[:, 2 + shift:, ev[b_]]
        y = t[:, 2:t.shape[1] - shift, ev[a]]
        d = x - y
        return float(np.nanmean(d)) / 1e3 if np.isfinite(d).any() else float("nan")

    def period(e):
        x = np.diff(t[:, 2:, ev[e]], axis=1)
        return float(np.nanmean(x)) / 1e3 if np.isfinite(x).any() else float("nan")

    # whole grid: first event and last epilogue completion per CTA
    starts, ends, ntiles = [], [], []
    for b in range(t.shape[0]):
        tb = t[b]
        if not np.isfinite(tb).any():
            continue
        starts.append(np.nanmin(tb))
        done = tb[:, ev["E_DONE"]]
        ends.append(np.nanmax(done) if np.isfinite(done).any() else np.nan)
        ntiles.append(int(np.isfinite(done).sum()))
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
    rows = [
        ("period per tile (M_EPI to M_EPI)", period("M_EPI")),
        ("K load: issue -> landed", span("P_ISSUE", "M_FULL")),
        ("stage empty wait -> loads issued", span("P_EMPTY", "P_ISSUE")),
        ("landed -> Gram issued", span("M_FULL", "M_GRAM")),
        ("Gram issued -> inverse starts", span("M_GRAM", "I_GRAM")),
        ("inverse: Gram ready -> T~ written", span("I_GRAM", "I_TT")),
        ("  wait for the previous T store to read", span("I_GRAM", "I_BW")),
        ("  Gram row load + L row", span("I_BW", "I_LD")),
        ("  16x16 diagonal substitution", span("I_LD", "I_DIAG")),
        ("  level-16 coupling", span("I_DIAG", "I_C16")),
        ("  pair sync", span("I_C16", "I_PAIR")),
        ("  level-32 coupling", span("I_PAIR", "I_INV")),
        ("  T store", span("I_INV", "I_TSTORE")),
        ("  wait T~ free", span("I_TSTORE", "I_TTW")),
        ("  write T~", span("I_TTW", "I_TT")),
        ("T~ written -> W|U MMA ready", span("I_TT", "M_READY")),
        ("W|U MMA ready -> issued", span("M_READY", "M_EPI")),
        ("W|U MMA issued -> epilogue starts", span("M_EPI", "E_DFULL")),
        ("epilogue: D loads", span("E_DFULL", "E_DEMPTY")),
        ("epilogue: total", span("E_DFULL", "E_DONE")),
        ("D drained -> next W|U MMA ready", span("E_DEMPTY", "M_READY", shift=1)),
        ("C=128: level-32 coupling", span("I_PAIR", "I_L32")),
        ("C=128: level-64 coupling", span("I_L32", "I_INV")),
        ("C=128: Gram ready -> level 32 ends, rows 0..63", span("I_GRAM", "I_L32")),
        ("C=128: Gram ready -> level 32 ends, rows 64..", span("I_GRAM", "I_L32B")),
        ("C=128: Gram ready -> M10 formed (epilogue)", span("I_GRAM", "E_M10")),
        ("C=128: level 32 end -> M00^-1 split, rows 0..", span("I_L32", "I_OPS")),
        ("C=128:   of which the stores are issued", span("I_L32", "I_SPLIT")),
        ("C=128: level 32 end -> M11^-1 in TMEM, 64..", span("I_L32B", "I_M11")),
        ("C=128: M00^-1 split -> Y issued", span("I_OPS", "M_L64Y")),
        ("C=128: Y issued -> Y seen by rows 64..", span("M_L64Y", "I_Y")),
        ("C=128: Y seen -> Y split to shared memory", span("I_Y", "I_YB")),
        ("C=128:   of which the stores are issued", span("I_Y", "I_YSPL")),
        ("C=128: Y split -> Z issued", span("I_YB", "M_L64Z")),
        ("C=128: Z issued -> Z seen by rows 64..", span("M_L64Z", "I_Z")),
        ("C=128: Z seen -> level 64 ends, rows 64..", span("I_Z", "I_INVB")),
        ("C=128: level 64 ends, rows 64.. -> rows 0..", span("I_INVB", "I_INV")),
    ]
    lines.append("")
    for name, val in rows:
        lines.append(f"{name:42s} {val:7.2f} us")
    return "\n".join(lines)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="c3_b4_t8192_h16")
    ap.add_argument("--ctas", type=int, default=2)
    ap.add_argument("--tiles", type=int, default=12)
    ap.add_argument("--static", action="store_true", help="fixed round-robin schedule (no workspace)")
    ap.add_argument("--save", default=None, help="also save the raw cycle counts (.npy)")
    ap.add_argument("--gated", action="store_true", help="the gated variant (seeded log decays)")
    ap.add_argument("--head-dim", type=int, default=None, help="override d_k = d_v (64 or 128)")
    a = ap.parse_args()
    tr = run(a.workload, dynamic=not a.static, gated=a.gated, head_dim=a.head_dim)
    print(f"untraced launch of the trace build: {run.last_ms * 1e3:.1f} us")
    print(report(tr, a.ctas, a.tiles))
    if a.save:
        np.save(a.save, run.last_raw)


if __name__ == "__main__":
    main()
