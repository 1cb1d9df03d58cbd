"""Comparison of library outputs with the fp64 oracle, and chunk bookkeeping for tests.

Tolerances (fixed by the spec contract of this library, written here):
  * T_out (fp32):            max |T - T_ref| <= 1e-4
  * W, U~ (bf16):            max |X - X_ref| <= 2e-2 where |X_ref| < 8, and
                             <= 2e-2 + half a bf16 ulp of X_ref where |X_ref| >= 8
                             (a bf16 value in [8, 16) is only resolved to 1/32);
                             relative Frobenius error <= 5e-3
  * W, U~ with fp32 I/O:     max |X - X_ref| <= 1e-4
The reference is always computed from the same bf16-rounded inputs.
"""
from __future__ import annotations

import math

import numpy as np
import torch

T_ATOL = 1e-4
WU_ATOL_BF16 = 2e-2
WU_RELFRO_BF16 = 5e-3
WU_ATOL_F32 = 1e-4


def chunks(C: int, B: int, T: int, cu_seqlens=None):
    """[(t0, Lc)] over the flat token axis, chunks restarting at every sequence start."""
    out = []
    if cu_seqlens is None:
        starts = [(b * T, (b + 1) * T) for b in range(B)]
    else:
        cu = [int(x) for x in cu_seqlens]
        starts = list(zip(cu[:-1], cu[1:]))
    for a, b in starts:
        for t0 in range(a, b, C):
            out.append((t0, min(C, b - t0)))
    return out


def _half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))  # bf16 keeps 8 significant bits


def check_T(T_gpu: np.ndarray, T_ref: np.ndarray, what="T"):
    err = np.abs(T_gpu.astype(np.float64) - T_ref)
    assert not np.isnan(T_gpu).any(), f"{what}: NaN"
    m = float(err.max()) if err.size else 0.0
    assert m <= T_ATOL, f"{what}: max abs error {m:.3e} > {T_ATOL}"
    return m


def check_WU(X_gpu: np.ndarray, X_ref: np.ndarray, io: str = "bf16", what="W"):
    X = X_gpu.astype(np.float64)
    assert not np.isnan(X).any(), f"{what}: NaN"
    err = np.abs(X - X_ref)
    if io == "f32":
        m = float(err.max()) if err.size else 0.0
        assert m <= WU_ATOL_F32, f"{what}: max abs error {m:.3e} > {WU_ATOL_F32}"
        return {"max_abs": m}
    big = np.abs(X_ref) >= 8.0
    small_max = float(err[~big].max()) if (~big).any() else 0.0
    assert small_max <= WU_ATOL_BF16, f"{what}: max abs error {small_max:.3e} > {WU_ATOL_BF16}"
    if big.any():
        lim = WU_ATOL_BF16 + _half_ulp_bf16(X_ref[big])
        assert np.all(err[big] <= lim), f"{what}: error above bf16 resolution at |x| >= 8"
    den = np.linalg.norm(X_ref)
    rel = float(np.linalg.norm(X - X_ref) / den) if den > 0 else float(np.linalg.norm(X))
    assert rel <= WU_RELFRO_BF16 or den == 0, f"{what}: relative Frobenius error {rel:.3e} > {WU_RELFRO_BF16}"
    return {"max_abs": small_max, "rel_fro": rel, "n_large": int(big.sum())}


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def relfro(a, b) -> float:
    d = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / d) if d > 0 else math.inf
