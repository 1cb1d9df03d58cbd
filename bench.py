#!/usr/bin/env python
"""Benchmark of kkt_solve fwd (chunk-local UT transform), one JSON line on stdout.

Workload (default): B=4 sequences x 8192 tokens = 32768 tokens, H=16 heads,
dk=dv=128, C=64, bf16 K/V/W/U, fp32 beta/T -- synthetic inputs (seeded; K rows
L2-normalised N(0,1), V ~ N(0,1), beta = sigmoid(N(0,1))).  A step is one call
of the whole path (A, T, W, U for every chunk and head).  The inputs (270 MB)
are larger than the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 launch one rank per GPU with torch.distributed.run; every rank runs
the same per-GPU workload (weak scaling, no collective on the data path) and
rank 0 prints the line with the max-over-ranks time.  ``--impl reference``
times the fp64 CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

import numpy as np
import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from gdn_chunkwise_ut_gb300 import costmodel  # noqa: E402
from gdn_chunkwise_ut_gb300.inputs import make_gate, workloads  # noqa: E402

METRIC = "tokens/sec and achieved HBM GB/s (% of GB300 peak) for kkt_solve fwd, C=64"
DEFAULT_WORKLOAD = "c3_b4_t8192_h16"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = {"simt": ["kkt_simt.cu", "kkt_internal.cuh", "kkt_debug.cuh"],
                  "tc": ["kkt_tc.cuh", "kkt_tc.cu", "sm100_ptx.cuh", "kkt_internal.cuh", "kkt_debug.cuh",
                         "tma_host.cuh"]}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "tc"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-pieces", type=int, default=8,
                    help="pieces the end-to-end runner pipelines each call in (copies in, kernel, copies out)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-t-out", action="store_true", help="W and U~ only: T computed, not written")
    ap.add_argument("--t-f16", action="store_true", help="T written in fp16 instead of fp32")
    ap.add_argument("--head-dim", type=int, default=None,
                    help="override the workload's head dimension d_k = d_v (64 or 128)")
    ap.add_argument("--dv", type=int, default=None,
                    help="override d_v alone, after --head-dim (mixed head dimensions)")
    ap.add_argument("--chunk", type=int, default=None,
                    help="override the workload's chunk size C (32, 64 or 128): the chunk-size study")
    ap.add_argument("--graph", action="store_true",
                    help="capture the K timed steps into one CUDA graph and time its replay")
    ap.add_argument("--gated", action="store_true",
                    help="gated variant: coefficient diag(beta)(Gamma o K K^T) from per-token log decays g")
    ap.add_argument("--no-consumer", dest="consumer", action="store_false",
                    help="skip timing the chunk state recurrence (gdn_chunk_state_fwd) that consumes W and U~, "
                         "and the two calls back to back, after the headline region")
    ap.add_argument("--consumer", dest="consumer", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.no_t_out and args.t_f16:
        ap.error("--no-t-out and --t-f16 exclude each other")
    return args


# --- distributed plumbing -------------------------------------------------------------------

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    return units_per_rank * world / max_seconds


# --- clocks ---------------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples (every 100 ms) of this GPU's SM clock and throttle reasons."""
    FIELDS = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.bus = None
        try:
            p = torch.cuda.get_device_properties(device_index)
            self.bus = f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
        except Exception:
            pass
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                if self.bus and parts[0].upper().lstrip("0") != self.bus.upper().lstrip("0"):
                    continue
                rows.append(parts)
        os.unlink(self.file.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for r in rows:
            try:
                sm.append(float(r[1])); mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --- peaks and recorded ncu traffic -----------------------------------------------------------

def hbm_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return float(json.loads(p.read_text())["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        h.update((ROOT / "gdn_chunkwise_ut_gb300" / "csrc" / name).read_bytes())
    return h.hexdigest()[:16]


def recorded_counters(kernel: str, workload: str) -> dict:
    """The committed ncu record of this kernel and workload (profiles/traffic.json), if it was taken
    from the current source; else {}."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return {}
    try:
        rec = json.loads(p.read_text()).get(f"{kernel}:{workload}")
    except Exception:
        return {}
    if not rec or rec.get("source_hash") != kernel_source_hash(kernel):
        return {}
    return rec


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source."""
    return recorded_counters(kernel, workload).get("dram_bytes_per_launch")


# --- our path -----------------------------------------------------------------------------------

def select_workload(args):
    w = workloads()[args.workload]
    if args.chunk is not None and args.chunk != w.C:
        w = dataclasses.replace(w, name=f"{w.name}@C{args.chunk}", C=args.chunk)
    if args.head_dim is not None and (args.head_dim != w.dk or args.head_dim != w.dv):
        w = dataclasses.replace(w, name=f"{w.name}@d{args.head_dim}", dk=args.head_dim, dv=args.head_dim)
    if args.dv is not None and args.dv != w.dv:
        w = dataclasses.replace(w, name=f"{w.name}@v{args.dv}", dv=args.dv)
    return w


def bench_ours(args, rank, world, local):
    from gdn_chunkwise_ut_gb300 import HostRunner, kkt_solve_fwd, select_kernel
    w = select_workload(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kernel = select_kernel(w.dk, w.dv, w.C, w.io, args.kernel)
    k, v, beta, cu = w.make(seed=rank, device=dev)
    g = make_gate(k.shape[0], k.shape[1], w.H, seed=rank, device=dev) if args.gated else None
    cu_t = None if cu is None else torch.as_tensor(cu, dtype=torch.int32, device=dev)
    T_dtype = torch.float16 if args.t_f16 else torch.float32
    T_out = torch.empty((k.shape[0], k.shape[1], w.H, w.C), device=dev, dtype=T_dtype)
    W_out = torch.empty_like(k)
    U_out = torch.empty_like(v)
    stream = torch.cuda.current_stream()

    def step():
        kkt_solve_fwd(k, v, beta, w.C, cu_t, T_out=None if args.no_t_out else T_out, W_out=W_out, U_out=U_out,
                      kernel=args.kernel, materialize_T=not args.no_t_out, T_dtype=T_dtype, g=g)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    # let the sampler see the GPU under load before the timed region
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 0.3:
        step()
        torch.cuda.synchronize()
    # Inputs larger than L2: K back-to-back steps between one pair of events on the launching
    # stream (events between the launches would add their own overhead to every step); the
    # per-launch duration the roofline uses is the region's average, so it includes the call's
    # workspace clear and launch gaps.  Inputs that fit in L2: every step gets its own events and
    # L2 is flushed before it (a write of twice its size, outside the events).
    K = args.steps
    in_bytes = sum(x.numel() * x.element_size() for x in (k, v, beta, g) if x is not None)
    flush = in_bytes <= L2_BYTES
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev) if flush else None
    barrier(world)
    torch.cuda.synchronize()
    if flush:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            scrub.zero_()
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        total_ms = sum(a.elapsed_time(b) for a, b in evs)
    elif args.graph:
        # the K steps as one CUDA graph (captured on a side stream after a warm-up there), replayed
        # once untimed and once between the events
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for i in range(K):
                step()
        graph.replay()
        torch.cuda.synchronize()
        t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        graph.replay()
        t_stop.record(stream)
        torch.cuda.synchronize()
        total_ms = t_start.elapsed_time(t_stop)
    else:
        t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(K):
            step()
        t_stop.record(stream)
        torch.cuda.synchronize()
        total_ms = t_start.elapsed_time(t_stop)
    barrier(world)
    clocks = sampler.stop()
    launch_ms = total_ms / K
    max_ms = max_over_ranks(total_ms, world)

    units = w.tokens * w.H
    io_bytes = 4 if w.io == "f32" else 2
    alg_bytes = units * costmodel.bytes_per_unit(w.C, w.dk, w.dv, io_bytes, t_out=not args.no_t_out,
                                                  t_bytes=2 if args.t_f16 else 4, gated=args.gated)
    tokens_per_s = aggregate_value(w.tokens * K, world, max_ms / 1e3)
    peak, peak_src = hbm_peak()
    achieved = alg_bytes / (launch_ms / 1e3) / 1e9
    # the recorded counters are those of the default call (fp32 T)
    # counters recorded for the default call and the gated one (fp32 T); none for the other variants
    counters = {} if (args.no_t_out or args.t_f16) else \
        recorded_counters(kernel, w.name + ("+gated" if args.gated else ""))
    traffic = counters.get("dram_bytes_per_launch")

    # end to end through the public API with host buffers (pinned), copies inside the timed region
    runner = HostRunner(k.shape[0], k.shape[1], w.H, w.dk, w.dv, w.C, dtype=k.dtype, cu_seqlens=cu,
                        kernel=args.kernel, device=dev, materialize_T=not args.no_t_out, T_dtype=T_dtype,
                        gated=args.gated, pieces=args.e2e_pieces)
    kh, vh, bh = (x.cpu().pin_memory() for x in (k, v, beta))
    gh = g.cpu().pin_memory() if g is not None else None
    for _ in range(2):
        runner(kh, vh, bh, g_host=gh)
    n_e2e = max(3, args.e2e_steps)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        runner(kh, vh, bh, g_host=gh)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e = {"value": aggregate_value(w.tokens * n_e2e, world, e2e_s), "unit": "tokens/s",
           "h2d_bytes_per_step": runner.h2d_bytes, "d2h_bytes_per_step": runner.d2h_bytes,
           "steps": n_e2e, "pieces": runner.pieces, "call": "kkt_solve_fwd_host"}

    # the specified entry point itself (kkt_solve_fwd: bf16, no workspace, so the tensor-core
    # kernel deals its tiles round robin), timed the same way on the same buffers, after the
    # timed region; reported beside the headline, which times the call with the workspace
    plain_call = None
    if w.io == "bf16" and not (args.no_t_out or args.t_f16 or args.gated or args.graph) and args.kernel == "auto":
        plain_call = time_kkt_solve_fwd_call(k, v, beta, cu_t, w, T_out, W_out, U_out, K, flush, scrub, stream)
        plain_call["headline_us_per_call"] = launch_ms * 1e3

    consumer = None
    if args.consumer:
        consumer = time_consumer(k, v, beta, g, cu_t, w, K, flush, scrub, stream, rank, peak)

    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": max_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.io == "bf16" else "f32",
        "data": "synthetic (seeded K rows L2-normalised N(0,1), V ~ N(0,1), beta = sigmoid(N(0,1)))",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                   "C": w.C, "tokens_per_step": w.tokens, "kernel": kernel,
                   "T_out": False if args.no_t_out else "fp16" if args.t_f16 else "fp32",
                   "gated": args.gated, "cuda_graph": bool(args.graph and not flush),
                   "l2": (f"inputs ({in_bytes / 1e6:.0f} MB) fit in the 129 MB L2: flushed before every step"
                          if flush else f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB > 129 MB), no flush")},
        "hbm_gbs": achieved, "hbm_frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
        "chunks_per_s": aggregate_value(units / w.C * K, world, max_ms / 1e3),
        # secondary: the tensor pipe's busy fraction from the committed ncu record (null when absent
        # or taken from other source)
        "tensor_pipe_active": counters.get("tensor_pipe_active"),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
                     "kernel": f"kkt_{kernel}", "alg_bytes_per_launch": alg_bytes,
                     "avg_launch_ms": launch_ms},
        "clocks": clocks, "e2e": e2e, "gpu_launches": K,
        "kkt_solve_fwd_call": plain_call,
        "gdn_chunk_state": consumer,
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(k, v, beta, cu, w, g=g)
    return line


def _device_time(fn, K, flush, scrub, stream):
    """Average device time (ms) of fn() over K calls: one event pair around K back-to-back calls, or,
    when the inputs fit in L2, per-call events with L2 flushed before each call."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    if flush:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            scrub.zero_()
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / K
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(K):
        fn()
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / K


def time_consumer(k, v, beta, g, cu_t, w, K, flush, scrub, stream, seed, peak):
    """gdn_chunk_state_fwd on the workload (W and U~ from kkt_solve, q and an initial state from the
    input recipe, the final state written), then kkt_solve and it back to back (the whole GDN forward
    of the chunked prefill)."""
    from gdn_chunkwise_ut_gb300 import gdn_chunk_state_fwd, kkt_solve_fwd
    from gdn_chunkwise_ut_gb300.inputs import make_query, make_state
    if w.dk != 128 or w.dv != 128 or w.C != 64 or w.io != "bf16":
        return {"skipped": "the recurrence kernel covers d_k = d_v = 128, C = 64, bf16"}
    dev = k.device
    q = make_query(k.shape[0], k.shape[1], w.H, w.dk, seed=seed, device=dev)
    N = w.B if cu_t is None else cu_t.shape[0] - 1
    S0 = make_state(N, w.H, w.dk, w.dv, seed=seed, device=dev)
    _, W, U = kkt_solve_fwd(k, v, beta, w.C, cu_t, materialize_T=False, g=g)
    o = torch.empty_like(v)
    S = torch.empty_like(S0)

    def rec():
        gdn_chunk_state_fwd(q, k, W, U, w.C, g=g, initial_state=S0, cu_seqlens=cu_t, o=o, final_state=S)

    def both():
        kkt_solve_fwd(k, v, beta, w.C, cu_t, T_out=None, W_out=W, U_out=U, materialize_T=False, g=g)
        rec()

    ms = _device_time(rec, K, flush, scrub, stream)
    ms_both = _device_time(both, K, flush, scrub, stream)
    units = w.tokens * w.H
    alg = units * costmodel.recurrence_bytes_per_unit(w.dk, w.dv, gated=g is not None) + \
        N * w.H * costmodel.state_bytes(w.dk, w.dv)
    gbs = alg / (ms / 1e3) / 1e9
    alg_both = alg + units * costmodel.bytes_per_unit(w.C, w.dk, w.dv, 2, t_out=False, gated=g is not None)
    return {"kernel": "gdn_chunk_kernel", "us_per_call": ms * 1e3, "tokens_per_s": w.tokens / (ms / 1e3),
            "alg_bytes_per_launch": alg, "hbm_gbs": gbs, "frac_of_peak": gbs / peak,
            "ctas": N * w.H, "chunks_per_cta": -(-max(w.T, max(w.lengths) if w.varlen else 0) // w.C),
            "with_kkt_solve_us": ms_both * 1e3, "with_kkt_solve_tokens_per_s": w.tokens / (ms_both / 1e3),
            "with_kkt_solve_gbs": alg_both / (ms_both / 1e3) / 1e9}


def time_kkt_solve_fwd_call(k, v, beta, cu_t, w, T_out, W_out, U_out, K, flush, scrub, stream):
    """Average device time of kkt_solve_fwd (the C entry point, through ctypes) over K calls."""
    from gdn_chunkwise_ut_gb300 import _lib
    lib = _lib.lib()
    B = w.B if cu_t is None else cu_t.shape[0] - 1
    args = (k.data_ptr(), v.data_ptr(), beta.data_ptr(), None if cu_t is None else cu_t.data_ptr(),
            B, k.shape[1], w.H, w.dk, w.dv, w.C, T_out.data_ptr(), W_out.data_ptr(), U_out.data_ptr(),
            stream.cuda_stream)
    for _ in range(3):
        rc = lib.kkt_solve_fwd(*args)
        if rc != _lib.KKT_OK:
            raise _lib.KktError(rc, "kkt_solve_fwd")
    torch.cuda.synchronize()
    if flush:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            scrub.zero_()
            evs[i][0].record(stream)
            lib.kkt_solve_fwd(*args)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        total_ms = sum(a.elapsed_time(b) for a, b in evs)
    else:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(K):
            lib.kkt_solve_fwd(*args)
        t1.record(stream)
        torch.cuda.synchronize()
        total_ms = t0.elapsed_time(t1)
    return {"entry": "kkt_solve_fwd", "schedule": "round robin (no workspace)",
            "us_per_call": total_ms / K * 1e3, "calls": K}


def cpu_baseline(k, v, beta, cu, w, max_tokens=None, g=None):
    """The oracle, as it stands, on the host cores over a bounded sample of the workload."""
    import oracle
    oracle.build()
    gs = None
    if cu is None:
        nseq = w.B if max_tokens is None else max(1, min(w.B, max_tokens // w.T))
        ks, vs, bs = (x[:nseq].cpu().double().numpy() for x in (k, v, beta))
        if g is not None:
            gs = g[:nseq].cpu().double().numpy()
        sample = f"{nseq} of {w.B} sequences x {w.T} tokens x {w.H} heads (fp64 oracle on bf16-rounded inputs)"
        tokens, cus = nseq * w.T, None
    else:
        ks, vs, bs = (x.cpu().double().numpy() for x in (k, v, beta))
        gs = None if g is None else g.cpu().double().numpy()
        tokens, cus, sample = w.tokens, cu, f"all {w.tokens} packed tokens x {w.H} heads"
    cores = oracle.oracle_threads(0)
    t0 = time.perf_counter()
    oracle.oracle_fwd(ks, vs, bs, w.C, cu_seqlens=cus, nthreads=cores, g=gs)
    dt = time.perf_counter() - t0
    out = {"value": tokens / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
           "sample": sample, "seconds": dt}
    if cu is None:
        # the same oracle on one core, over one sequence and up to 4 heads, as tokens/s of all H heads
        hs = min(w.H, 4)
        k1, v1, b1 = (np.ascontiguousarray(x[:1, :, :hs]) for x in (ks, vs, bs))
        g1 = None if gs is None else np.ascontiguousarray(gs[:1, :, :hs])
        t0 = time.perf_counter()
        oracle.oracle_fwd(k1, v1, b1, w.C, nthreads=1, g=g1)
        dt1 = time.perf_counter() - t0
        out["one_core"] = {"value": w.T * hs / w.H / dt1, "unit": "tokens/s",
                           "sample": f"1 sequence x {w.T} tokens x {hs} of {w.H} heads, 1 thread",
                           "seconds": dt1}
    return out


# --- reference arm: the oracle on the host cores -----------------------------------------------

def bench_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    w = select_workload(args)
    if w.varlen:
        raise SystemExit("reference arm covers fixed-length workloads")
    # each step: one chunk-aligned slice of one sequence, all heads, sized so that
    # warmup + steps fit in about two minutes of wall time
    from gdn_chunkwise_ut_gb300.inputs import make_inputs
    cores = oracle.oracle_threads(0)
    probe_tokens = w.C * 4
    k, v, b = make_inputs(1, probe_tokens, w.H, w.dk, w.dv, seed=0)
    kd, vd, bd = (x.double().numpy() for x in (k, v, b))
    gd = make_gate(1, probe_tokens, w.H, seed=0).double().numpy() if args.gated else None
    t0 = time.perf_counter()
    oracle.oracle_fwd(kd, vd, bd, w.C, nthreads=cores, g=gd)
    per_token = (time.perf_counter() - t0) / probe_tokens
    budget = 120.0 / max(1, args.steps + args.warmup)
    tokens = int(max(w.C, min(w.T, (budget / per_token) // w.C * w.C)))
    k, v, b = make_inputs(1, tokens, w.H, w.dk, w.dv, seed=0)
    kd, vd, bd = (x.double().numpy() for x in (k, v, b))
    gd = make_gate(1, tokens, w.H, seed=0).double().numpy() if args.gated else None
    for _ in range(args.warmup):
        oracle.oracle_fwd(kd, vd, bd, w.C, nthreads=cores, g=gd)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.oracle_fwd(kd, vd, bd, w.C, nthreads=cores, g=gd)
    dt = time.perf_counter() - t0
    val = tokens * args.steps / dt
    sample = f"{tokens} tokens x {w.H} heads of one {w.T}-token sequence per step (fp64 oracle)"
    return {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H,
                                        "dk": w.dk, "dv": w.dv, "C": w.C, "tokens_per_step": tokens,
                                        "gated": args.gated},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    args = parse_args()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        line = bench_reference(args, rank, world)
    else:
        line = bench_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
