"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

from gdn_chunkwise_ut_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(kkt_\w+)\s*\(", text))
    return sorted(names)


def test_workspace_size_constant_matches_header():
    text = open(os.path.join(ROOT, "include", "kkt.h")).read()
    m = re.search(r"#define\s+KKT_WORKSPACE_BYTES\s+(\d+)", text)
    assert m and int(m.group(1)) == _lib.KKT_WORKSPACE_BYTES
    m = re.search(r"#define\s+KKT_T_OUT_F16\s+(0x[0-9a-fA-F]+)", text)
    assert m and int(m.group(1), 16) == _lib.KKT_T_OUT_F16


def test_trace_tool_matches_the_kernels_event_table():
    """The trace tool decodes the kernel's trace buffer by the order of its event enum and by its
    row size; both sides are written by hand, so a drift would mislabel every event."""
    from gdn_chunkwise_ut_gb300 import trace
    text = open(os.path.join(ROOT, "gdn_chunkwise_ut_gb300", "csrc", "kkt_tc.cuh")).read()
    body = re.search(r"enum TraceEvent \{(.*?)\};", text, flags=re.S).group(1)
    body = re.sub(r"//[^\n]*", "", body)
    names = [n.strip().split("=")[0].strip() for n in body.split(",") if n.strip()]
    assert names[-1] == "EV_COUNT"
    assert [n[len("EV_"):] for n in names[:-1]] == trace.EVENTS
    slots = int(re.search(r"constexpr int kTraceSlots = (\d+);", text).group(1))
    tiles = int(re.search(r"constexpr int kTraceTiles = (\d+);", text).group(1))
    ctas = int(re.search(r"constexpr int kTraceCtas = (\d+);", text).group(1))
    assert (trace.TRACE_CTAS, trace.TRACE_TILES, trace.TRACE_SLOTS) == (ctas, tiles, slots)
    assert len(trace.EVENTS) <= slots


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "kkt_solve_fwd" in names and "kkt_solve_fwd_ex" in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature"


def test_no_cuda_shared_library_dependency():
    """Static cudart and a driver entry point looked up at run time: loads without a GPU."""
    import subprocess
    out = subprocess.run(["ldd", str(_lib.LIB_PATH)], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libcudart.so" not in out


def test_status_strings_and_version(lib):
    for s in range(8):
        assert lib.kkt_status_string(s).decode() != "unknown status"
    assert lib.kkt_status_string(99).decode() == "unknown status"
    assert lib.kkt_version() >= (0 << 16) | (1 << 8)


def test_select_kernel(lib):
    sel = lib.kkt_select_kernel
    assert sel(128, 128, 64, _lib.KKT_IO_F32, _lib.KKT_KERNEL_AUTO) == _lib.KKT_KERNEL_SIMT
    assert sel(128, 128, 64, _lib.KKT_IO_F32, _lib.KKT_KERNEL_TC) == -_lib.KKT_ERR_UNSUPPORTED
    assert sel(128, 128, 64, _lib.KKT_IO_BF16, _lib.KKT_KERNEL_SIMT) == _lib.KKT_KERNEL_SIMT
    assert sel(96, 128, 64, _lib.KKT_IO_BF16, 0) == -_lib.KKT_ERR_UNSUPPORTED
    assert sel(128, 128, 48, _lib.KKT_IO_BF16, 0) == -_lib.KKT_ERR_UNSUPPORTED
    assert sel(128, 128, 256, _lib.KKT_IO_BF16, 0) == -_lib.KKT_ERR_UNSUPPORTED
    assert sel(128, 128, 64, 7, 0) == -_lib.KKT_ERR_ARG
    assert sel(128, 128, 64, _lib.KKT_IO_BF16, 9) == -_lib.KKT_ERR_ARG
    # the precision of T_out does not change the kernel chosen
    assert sel(128, 128, 64, _lib.KKT_IO_BF16 | _lib.KKT_T_OUT_F16, 0) == _lib.KKT_KERNEL_TC
    assert sel(128, 128, 64, _lib.KKT_IO_F32 | _lib.KKT_T_OUT_F16, 0) == _lib.KKT_KERNEL_SIMT
    assert sel(128, 128, 64, 0x200, 0) == -_lib.KKT_ERR_ARG
    for C in (32, 64, 128):
        for dk in (64, 128):
            for dv in (64, 128):
                # the tensor-core kernel covers every bf16 shape (d_k = d_v or not); fp32 I/O runs
                # on the SIMT kernel only, which also takes every bf16 shape when asked for
                assert sel(dk, dv, C, _lib.KKT_IO_BF16, _lib.KKT_KERNEL_AUTO) == _lib.KKT_KERNEL_TC
                assert sel(dk, dv, C, _lib.KKT_IO_BF16, _lib.KKT_KERNEL_SIMT) == _lib.KKT_KERNEL_SIMT
                assert sel(dk, dv, C, _lib.KKT_IO_F32, _lib.KKT_KERNEL_AUTO) == _lib.KKT_KERNEL_SIMT
                assert sel(dk, dv, C, _lib.KKT_IO_F32, _lib.KKT_KERNEL_TC) == -_lib.KKT_ERR_UNSUPPORTED


def _call(lib, **kw):
    a = dict(k=0x1000, v=0x2000, beta=0x3000, cu=None, B=1, T=64, H=1, dk=128, dv=128, C=64,
             T_out=0x4000, W_out=0x5000, U_out=0x6000, io=0, kernel=0, ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.kkt_solve_fwd_ex(a["k"], a["v"], a["beta"], a["cu"], a["B"], a["T"], a["H"], a["dk"],
                                a["dv"], a["C"], a["T_out"], a["W_out"], a["U_out"], a["io"],
                                a["kernel"], a["ws"], a["ws_bytes"], a["stream"])


def test_argument_errors_return_before_launch(lib):
    """None of these reach CUDA: the addresses are never dereferenced."""
    assert _call(lib, k=None) == _lib.KKT_ERR_ARG
    assert _call(lib, U_out=None) == _lib.KKT_ERR_ARG
    assert _call(lib, B=0) == _lib.KKT_ERR_ARG
    assert _call(lib, T=-1) == _lib.KKT_ERR_ARG
    assert _call(lib, H=0) == _lib.KKT_ERR_ARG
    assert _call(lib, H=70000) == _lib.KKT_ERR_ARG
    assert _call(lib, dk=96) == _lib.KKT_ERR_UNSUPPORTED
    assert _call(lib, C=16) == _lib.KKT_ERR_UNSUPPORTED
    assert _call(lib, io=3) == _lib.KKT_ERR_ARG
    assert _call(lib, io=1, kernel=2) == _lib.KKT_ERR_UNSUPPORTED
    assert _call(lib, k=0x1008) == _lib.KKT_ERR_ALIGN
    assert _call(lib, W_out=0x5004) == _lib.KKT_ERR_ALIGN
    assert _call(lib, cu=0x7002) == _lib.KKT_ERR_ALIGN
    assert _call(lib, beta=0x3002) == _lib.KKT_ERR_ALIGN
    assert _call(lib, ws=0x8000, ws_bytes=_lib.KKT_WORKSPACE_BYTES - 1) == _lib.KKT_ERR_ARG
    assert _call(lib, ws=0x8004, ws_bytes=_lib.KKT_WORKSPACE_BYTES) == _lib.KKT_ERR_ALIGN
    assert _call(lib, T=0) == _lib.KKT_OK               # empty batch: nothing to launch
    assert _call(lib, T_out=None, T=0) == _lib.KKT_OK   # T_out may be NULL (W and U~ only)
    assert _call(lib, T_out=0x4004) == _lib.KKT_ERR_ALIGN
    assert _call(lib, T_out=0x4004, io=_lib.KKT_T_OUT_F16) == _lib.KKT_ERR_ALIGN
    assert _call(lib, io=0x200) == _lib.KKT_ERR_ARG
    assert _call(lib, T=0, io=_lib.KKT_T_OUT_F16) == _lib.KKT_OK
    assert _call(lib, cu=0x7000, B=3, T=0) == _lib.KKT_OK
    assert lib.kkt_solve_fwd(None, 0x2000, 0x3000, None, 1, 64, 1, 128, 128, 64,
                             0x4000, 0x5000, 0x6000, None) == _lib.KKT_ERR_ARG


def test_gated_argument_errors(lib):
    """The gated entry point checks g like beta (4-byte aligned) and otherwise as kkt_solve_fwd_ex."""
    def call(g=0x9000, **kw):
        a = dict(k=0x1000, v=0x2000, beta=0x3000, T=64, C=64, T_out=0x4000)
        a.update(kw)
        return lib.kkt_solve_fwd_gated(a["k"], 0x2000, a["beta"], g, None, 1, a["T"], 1, 128, 128, a["C"],
                                       a["T_out"], 0x5000, 0x6000, 0, 0, None, 0, None)
    assert call(g=0x9002) == _lib.KKT_ERR_ALIGN
    assert call(k=None) == _lib.KKT_ERR_ARG
    assert call(C=48) == _lib.KKT_ERR_UNSUPPORTED
    assert call(T=0) == _lib.KKT_OK
    assert call(g=None, T=0) == _lib.KKT_OK  # g == NULL is the ungated call


def test_default_build_has_no_bounds_checks(lib):
    """kkt_debug_bounds reports -1 in the default build: no checks are compiled into the product."""
    assert lib.kkt_debug_bounds(None, None) == -1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """The product path has no fallback: without libkkt.so every call raises."""
    monkeypatch.setattr(_lib, "LIB_PATH", tmp_path / "libkkt.so")
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.lib()


def test_ctypes_signature_arity():
    for name, (_, args) in _lib.SIGNATURES.items():
        assert all(a in (ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float) for a in args), name
