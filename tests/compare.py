"""Comparison of library outputs with the fp64 oracle, and chunk bookkeeping for tests.

Tolerances (fixed by the accuracy contract of this library's specification, written here):
  * T_out (fp32):            max |T - T_ref| <= 1e-4
  * W, U~ (bf16):            max |X - X_ref| <= 2e-2 where |X_ref| < 8, and
                             <= 2e-2 + half a bf16 ulp of X_ref where |X_ref| >= 8
                             (a bf16 value in [8, 16) is only resolved to 1/32);
                             relative Frobenius error <= 5e-3
  * W, U~ with fp32 I/O:     max |X - X_ref| <= 1e-4
The reference is always computed from the same bf16-rounded inputs.

The chunk state recurrence and output (gdn_chunk_state_fwd), whose products round three operands
to bf16 (the state S, V' and the masked Q K^T) besides the output, against the fp64 oracle:
  * o (bf16):                max-abs <= 2e-2, relative Frobenius <= 1e-2
  * final state (fp32):      max-abs <= 5e-2, relative Frobenius <= 1e-2
(a numpy emulation of those rounding points gives about 3e-3 and 2.5e-3 relative Frobenius on
o and the state, with o's entries below 0.4 and the state's below 3).
"""
from __future__ import annotations

import math

import numpy as np
import torch

T_ATOL = 1e-4
WU_ATOL_BF16 = 2e-2
WU_RELFRO_BF16 = 5e-3
WU_ATOL_F32 = 1e-4
O_ATOL = 2e-2
O_RELFRO = 1e-2
STATE_ATOL = 5e-2
STATE_RELFRO = 1e-2


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


def check_recurrence(o_gpu: np.ndarray, o_ref: np.ndarray, s_gpu=None, s_ref=None, what=""):
    """Output and final state of the chunk recurrence against the oracle; returns the errors."""
    out = {}
    for name, X, R, atol, rtol in (("o", o_gpu, o_ref, O_ATOL, O_RELFRO), ("state", s_gpu, s_ref, STATE_ATOL, STATE_RELFRO)):
        if X is None:
            continue
        X = X.astype(np.float64)
        assert not np.isnan(X).any(), f"{what}{name}: NaN"
        m = float(np.abs(X - R).max()) if X.size else 0.0
        den = np.linalg.norm(R)
        rel = float(np.linalg.norm(X - R) / den) if den > 0 else float(np.linalg.norm(X))
        assert m <= atol, f"{what}{name}: max abs error {m:.3e} > {atol}"
        assert rel <= rtol, f"{what}{name}: relative Frobenius error {rel:.3e} > {rtol}"
        out[f"{name}_max_abs"], out[f"{name}_rel_fro"] = m, rel
    return out


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def relfro(a, b) -> float:
    d = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / d) if d > 0 else math.inf


class FullComparison:
    """Whole-tensor comparison of T, W and U~ with the oracle, accumulated slab by slab.

    A slab is a group of whole sequences; the oracle runs on each slab on its own (its chunks never
    cross a sequence start, so that is the oracle of the whole batch), and the library's outputs
    for the slab are compared with it element by element under the tolerances above.  The relative
    Frobenius error is accumulated over the whole tensor.  ``n_large`` counts the W / U~ elements
    with |x_ref| >= 8, whose bound is widened by half a bf16 ulp.
    """

    def __init__(self, io: str = "bf16"):
        self.io = io
        self.T_max = 0.0
        self.stats = {n: {"max_abs": 0.0, "err2": 0.0, "ref2": 0.0, "n_large": 0, "n": 0} for n in ("W", "U")}

    def add(self, T_gpu, W_gpu, U_gpu, T_ref, W_ref, U_ref):
        if T_gpu is not None:
            self.T_max = max(self.T_max, check_T(T_gpu, T_ref))
        for name, X, R in (("W", W_gpu, W_ref), ("U", U_gpu, U_ref)):
            X = X.astype(np.float64)
            assert not np.isnan(X).any(), f"{name}: NaN"
            err = np.abs(X - R)
            st = self.stats[name]
            st["n"] += err.size
            st["err2"] += float(np.square(X - R).sum())
            st["ref2"] += float(np.square(R).sum())
            if self.io == "f32":
                m = float(err.max()) if err.size else 0.0
                assert m <= WU_ATOL_F32, f"{name}: max abs error {m:.3e} > {WU_ATOL_F32}"
                st["max_abs"] = max(st["max_abs"], m)
                continue
            big = np.abs(R) >= 8.0
            small_max = float(err[~big].max()) if (~big).any() else 0.0
            assert small_max <= WU_ATOL_BF16, f"{name}: max abs error {small_max:.3e} > {WU_ATOL_BF16}"
            if big.any():
                lim = WU_ATOL_BF16 + _half_ulp_bf16(R[big])
                assert np.all(err[big] <= lim), f"{name}: error above bf16 resolution at |x| >= 8"
                st["max_abs"] = max(st["max_abs"], float(err[big].max()))
            st["max_abs"] = max(st["max_abs"], small_max)
            st["n_large"] += int(big.sum())

    def finish(self) -> dict:
        out = {"T_max_abs": self.T_max}
        for name, st in self.stats.items():
            rel = math.sqrt(st["err2"] / st["ref2"]) if st["ref2"] > 0 else math.sqrt(st["err2"])
            if self.io != "f32":
                assert rel <= WU_RELFRO_BF16, f"{name}: relative Frobenius error {rel:.3e} > {WU_RELFRO_BF16}"
            out[f"{name}_max_abs"] = st["max_abs"]
            out[f"{name}_rel_fro"] = rel
            out[f"{name}_n_large"] = st["n_large"]
            out[f"{name}_elements"] = st["n"]
        return out


def slabs(B: int, T: int, cu_seqlens=None, max_tokens: int = 16384):
    """Groups of whole sequences [(n0, n1, cu_rel or None)] on the flat token axis, each of about
    ``max_tokens`` tokens or one sequence."""
    if cu_seqlens is None:
        per = max(1, max_tokens // max(T, 1))
        return [(b * T, min(B, b + per) * T, None) for b in range(0, B, per)]
    cu = [int(x) for x in cu_seqlens]
    out, s = [], 0
    while s < len(cu) - 1:
        e = s + 1
        while e < len(cu) - 1 and cu[e + 1] - cu[s] <= max_tokens:
            e += 1
        out.append((cu[s], cu[e], np.asarray([c - cu[s] for c in cu[s:e + 1]], dtype=np.int64)))
        s = e
    return out
