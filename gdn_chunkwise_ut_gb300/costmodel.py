"""Cost model of the blocked unit-lower-triangular inverse and of the kkt_solve path.

Pure arithmetic on sizes (no tensors): FMA counts and dependency-chain lengths
of the schedule the CUDA kernels run, and the algorithmic bytes / MACs per
(token, head) unit that the roofline figures in ``bench.py`` divide by.

The schedule ("TileLang 实战：单位下三角矩阵求逆" §2.2-§2.3): split the C x C
unit lower-triangular matrix into 16 x 16 diagonal blocks, invert each by
row forward substitution (§2.1: n(n-1)(n-2)/6 FMA in n-1 dependent steps),
then couple neighbouring inverses level by level, s = 16, 32, ..., C/2, with
two s x s x s GEMMs per pair (-L11^-1 L10 L00^-1), each level adding two
dependent steps.  The tests check these formulas against the figures the page
prints (§2.2 method table, §2.3 tables, §2.4 tables).
"""
from __future__ import annotations

BASE = 16  # size of the diagonal blocks inverted by substitution


def row_fma(n: int) -> int:
    """FMA of element-wise forward substitution of an n x n unit lower-triangular inverse."""
    return n * (n - 1) * (n - 2) // 6


def row_chain(n: int) -> int:
    """Dependent steps of element-wise forward substitution (one per row after the first)."""
    return n - 1


def levels(C: int, base: int = BASE) -> int:
    """Recursion depth: number of coupling levels between base and C."""
    d, s = 0, base
    while s < C:
        s *= 2
        d += 1
    if s != C:
        raise ValueError(f"C={C} is not base * 2^d")
    return d


def coupling_pairs(C: int, base: int = BASE) -> list:
    """[(s, pairs at that level)] for s = base, 2 base, ..., C/2."""
    out, s = [], base
    while s < C:
        out.append((s, C // (2 * s)))
        s *= 2
    return out


def blocked_fma(C: int, base: int = BASE) -> int:
    """FMA of the blocked recursion: C/base substitutions + 2 s^3 per coupling pair."""
    return (C // base) * row_fma(base) + sum(p * 2 * s ** 3 for s, p in coupling_pairs(C, base))


def blocked_chain(C: int, base: int = BASE) -> int:
    """Dependent steps: base-1 for the substitutions, +2 per coupling level."""
    return row_chain(base) + 2 * levels(C, base)


def flat_block_gemms(C: int, base: int = BASE) -> int:
    """base^3 GEMMs of flat block substitution on the (C/base)^2 grid.

    Block row r, block column j < r: X[r][j] = -X[r][r] * sum_{m=j}^{r-1} L[r][m] X[m][j],
    i.e. (r - j) GEMMs for the sum and one for the product with X[r][r].
    """
    nb = C // base
    return sum(r - j + 1 for r in range(1, nb) for j in range(r))


def flat_block_fma(C: int, base: int = BASE) -> int:
    return (C // base) * row_fma(base) + flat_block_gemms(C, base) * base ** 3


def flat_block_chain(C: int, base: int = BASE) -> int:
    """base-1 substitution steps, then two dependent GEMM steps per later block row."""
    return row_chain(base) + 2 * (C // base - 1)


def stage_table(C: int, base: int = BASE) -> list:
    """[(independent tasks, added depth, parallel output elements)] per stage."""
    rows = [(C // base, row_chain(base), (C // base) * base)]
    for s, p in coupling_pairs(C, base):
        rows.append((p, 2, p * s * s))
    return rows


def main_gemm_per_token(C: int, dk: int, dv: int) -> int:
    """Per-token MACs of the chunkwise main GEMMs: 2 dk dv + C (dk + dv) (§2.4)."""
    return 2 * dk * dv + C * (dk + dv)


def bytes_per_unit(C: int, dk: int, dv: int, io_bytes: int = 2, t_out: bool = True, t_bytes: int = 4,
                   gated: bool = False) -> int:
    """Algorithmic HBM bytes per (token, head): read K, V, beta (and the fp32 log decay g when
    gated); write T (t_bytes per element: 4 for fp32, 2 for fp16; nothing when the call produces
    W and U only), W, U."""
    return io_bytes * (dk + dv) + 4 + (4 if gated else 0) + (t_bytes * C if t_out else 0) + io_bytes * (dk + dv)


def bytes_written_per_unit(C: int, dk: int, dv: int, io_bytes: int = 2) -> int:
    return 4 * C + io_bytes * (dk + dv)


def triangular_mac_per_unit(C: int, dk: int, dv: int) -> float:
    """MACs per (token, head) that the method needs, counting only nonzero triangles."""
    gram = (C - 1) / 2 * dk
    inverse = blocked_fma(C) / C
    epilogue = (C + 1) / 2 * (dk + dv)
    return gram + inverse + epilogue


def recurrence_bytes_per_unit(dk: int, dv: int, gated: bool = False) -> int:
    """Algorithmic HBM bytes per (token, head) of the chunk state recurrence and output: read q, k, W
    (bf16, d_k each) and U~ (bf16, d_v), the gate's log decay (fp32) when gated; write o (bf16, d_v)."""
    return 2 * (3 * dk + dv) + 2 * dv + (4 if gated else 0)


def state_bytes(dk: int, dv: int) -> int:
    """Bytes per (sequence, head) of the recurrence's fp32 states: the initial one read, the final one
    written."""
    return 2 * 4 * dk * dv
