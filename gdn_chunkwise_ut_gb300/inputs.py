"""Seeded synthetic inputs for kkt_solve (shared by tests, bench and smoke).

This module holds only the input recipe -- no step of the UT transform.  Both
the CUDA path and the CPU oracle are fed from it; neither imports the other.

Recipe (the five benchmark configurations of the library's specification; the pages' own
benchmark runs on Qwen3.5/3.6 head configurations, h_v in {64,48,32,24,16,8},
per the FlashQLA announcement's Benchmark section, and these synthetic tensors
stand in for that data):
  * K: rows ~ N(0, 1) in fp32, L2-normalised along d_k (the pages state that k
    is L2-normalised upstream of the kernel, "TileLang 实战：单位下三角矩阵求逆"
    §1), then rounded to the I/O dtype (bf16, or fp32 for the small case);
  * V: N(0, 1) rounded to the I/O dtype;
  * beta: sigmoid(N(0, 1)) in fp32, so beta in (0, 1) (§1: the write strength);
  * g (gated variant only): log sigmoid(N(2.5, 1)) in fp32, a per-token log decay with
    alpha = exp(g) in (0, 1) (the FlashQLA page's gate, "Gate 衰减性质" section), mean decay
    about 0.9 per token, so that Gamma falls to about e^-6 across a 64-token chunk.
  * q (the chunk recurrence): rows ~ N(0, 1), L2-normalised like K, rounded to bf16;
  * initial state (the chunk recurrence): N(0, 1) / sqrt(d_k) in fp32.
Variable-length batches draw 32 lengths uniform in [100, 8192] with
``numpy.random.default_rng(1234)``.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


def make_inputs(B: int, T: int, H: int, dk: int, dv: int, *, seed: int = 0,
                dtype: torch.dtype = torch.bfloat16, device="cpu"):
    """k [B,T,H,dk], v [B,T,H,dv] in ``dtype``; beta [B,T,H] fp32."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    k = torch.randn((B, T, H, dk), generator=g, device=device, dtype=torch.float32)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    v = torch.randn((B, T, H, dv), generator=g, device=device, dtype=torch.float32)
    beta = torch.sigmoid(torch.randn((B, T, H), generator=g, device=device, dtype=torch.float32))
    return k.to(dtype).contiguous(), v.to(dtype).contiguous(), beta.contiguous()


def make_gate(B: int, T: int, H: int, *, seed: int = 0, device="cpu"):
    """g [B,T,H] fp32: per-token log decays log sigmoid(N(2.5, 1)), all < 0."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 7919)
    x = torch.randn((B, T, H), generator=gen, device=device, dtype=torch.float32) + 2.5
    return torch.nn.functional.logsigmoid(x).contiguous()


def make_query(B: int, T: int, H: int, dk: int, *, seed: int = 0, device="cpu"):
    """q [B,T,H,dk] bf16: rows ~ N(0, 1), L2-normalised like the keys (the recurrence's queries)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 104729)
    q = torch.randn((B, T, H, dk), generator=gen, device=device, dtype=torch.float32)
    return (q / q.norm(dim=-1, keepdim=True).clamp_min(1e-12)).to(torch.bfloat16).contiguous()


def make_state(N: int, H: int, dk: int, dv: int, *, seed: int = 0, device="cpu"):
    """An initial state [N,H,dk,dv] fp32: N(0, 1) / sqrt(dk), about the size the recurrence keeps."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 1299709)
    return (torch.randn((N, H, dk, dv), generator=gen, device=device, dtype=torch.float32) * dk ** -0.5).contiguous()


def varlen_lengths(n: int = 32, lo: int = 100, hi: int = 8192, seed: int = 1234) -> np.ndarray:
    """Sequence lengths uniform in [lo, hi] (inclusive), seed-fixed."""
    return np.random.default_rng(seed).integers(lo, hi + 1, n).astype(np.int64)


def cu_seqlens_from_lengths(lengths) -> np.ndarray:
    lengths = np.asarray(lengths, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, chunk size and I/O dtype."""
    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    C: int
    io: str = "bf16"                      # "bf16" or "f32"
    lengths: tuple = field(default=())    # non-empty -> varlen, tensors [1, sum, H, .]

    @property
    def varlen(self) -> bool:
        return len(self.lengths) > 0

    @property
    def tokens(self) -> int:
        return int(sum(self.lengths)) if self.varlen else self.B * self.T

    @property
    def torch_dtype(self):
        return torch.float32 if self.io == "f32" else torch.bfloat16

    def cu_seqlens(self):
        return cu_seqlens_from_lengths(self.lengths) if self.varlen else None

    def make(self, seed: int = 0, device="cpu"):
        """(k, v, beta, cu_seqlens or None) with the tensor shapes the library takes."""
        if self.varlen:
            k, v, beta = make_inputs(1, self.tokens, self.H, self.dk, self.dv, seed=seed,
                                     dtype=self.torch_dtype, device=device)
            return k, v, beta, self.cu_seqlens()
        k, v, beta = make_inputs(self.B, self.T, self.H, self.dk, self.dv, seed=seed,
                                 dtype=self.torch_dtype, device=device)
        return k, v, beta, None


def workloads() -> dict:
    """The five workload families, expanded into named single runs."""
    w = {
        # single head, one 128-token sequence, C=32 (4 chunks), dk=dv=64, fp32 I/O
        "c1_small_f32": Workload("c1_small_f32", 1, 128, 1, 64, 64, 32, io="f32"),
        # one 8192-token sequence, 16 heads, C=64
        "c2_t8192_h16": Workload("c2_t8192_h16", 1, 8192, 16, 128, 128, 64),
    }
    # four 8192-token sequences (32768 tokens), head-count sweep, C=64
    for H in (64, 48, 32, 24, 16, 8):
        w[f"c3_b4_t8192_h{H}"] = Workload(f"c3_b4_t8192_h{H}", 4, 8192, H, 128, 128, 64)
    # 32 packed sequences, lengths uniform in [100, 8192], 32 heads, C=64
    w["c4_varlen32_h32"] = Workload("c4_varlen32_h32", 32, 0, 32, 128, 128, 64,
                                    lengths=tuple(int(x) for x in varlen_lengths()))
    # chunk-size study: two 16384-token sequences, 24 heads, C in {32, 64, 128}
    for C in (32, 64, 128):
        w[f"c5_b2_t16384_h24_c{C}"] = Workload(f"c5_b2_t16384_h24_c{C}", 2, 16384, 24, 128, 128, C)
    return w
