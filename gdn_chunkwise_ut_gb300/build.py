"""Builds libkkt.so in-tree with nvcc for sm_103a (GB300).

One ``nvcc -c`` per translation unit, run in parallel, then one ``nvcc -shared``
link.  The CUDA runtime is linked statically and the CUDA driver is reached
through ``cudaGetDriverEntryPointByVersion``, so the library loads on a machine
without a GPU (the ABI tests rely on that).
"""
from __future__ import annotations

import os
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIB = BUILD / "libkkt.so"
INCLUDE = ROOT / "include"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "-Xptxas", "-v", "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources() -> list:
    return sorted(CSRC.glob("*.cu"))


def _stale(out: Path, deps) -> bool:
    if not out.exists():
        return True
    t = out.stat().st_mtime
    return any(Path(d).stat().st_mtime > t for d in deps)


def build(verbose: bool = False, force: bool = False, extra_flags=(), trace: bool = False,
          debug_bounds: bool = False) -> Path:
    """Compile every csrc/*.cu and link libkkt.so; returns the library path.

    ``trace=True`` builds a separate libkkt_trace.so (in _build/trace) with the
    pipeline time stamps of the tensor-core kernel compiled in (see trace.py).
    ``debug_bounds=True`` builds a separate libkkt_bounds.so (in _build/bounds) with
    every shared-memory, array and plain global access range-checked (kkt_debug.cuh;
    read with kkt_debug_bounds()).
    """
    if trace and debug_bounds:
        raise ValueError("trace and debug_bounds are separate builds")
    out_dir = BUILD / "trace" if trace else BUILD / "bounds" if debug_bounds else BUILD
    lib_path = out_dir / ("libkkt_trace.so" if trace else "libkkt_bounds.so" if debug_bounds else "libkkt.so")
    if trace:
        extra_flags = (*extra_flags, "-DKKT_TRACE")
    if debug_bounds:
        extra_flags = (*extra_flags, "-DKKT_DEBUG_BOUNDS")
    out_dir.mkdir(parents=True, exist_ok=True)
    headers = list(CSRC.glob("*.cuh")) + list(INCLUDE.glob("*.h"))
    nvcc = _nvcc()
    procs, objs = [], []
    for src in sources():
        obj = out_dir / (src.stem + ".o")
        objs.append(obj)
        if force or _stale(obj, [src, *headers]):
            log = out_dir / (src.stem + ".log")
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", str(src), "-o", str(obj)]
            procs.append((src, log, subprocess.Popen(cmd, stdout=open(log, "w"), stderr=subprocess.STDOUT)))
    failed = []
    for src, log, p in procs:
        if p.wait() != 0:
            failed.append((src, log))
        elif verbose:
            sys.stdout.write(log.read_text())
    if failed:
        msg = "\n".join(f"--- {s.name} ---\n{l.read_text()}" for s, l in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    if force or _stale(lib_path, objs):
        tmp = out_dir / f"libkkt.{os.getpid()}.tmp.so"
        cmd = [nvcc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":  # pragma: no cover
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
