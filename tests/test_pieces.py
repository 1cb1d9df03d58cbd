"""The piece planner of kkt_solve_fwd_host (host logic in the C library, no GPU): the pieces tile the
token axis in order, there are never more than asked for, every cut inside a sequence falls on a
chunk boundary of that sequence, and each piece's sequence offsets describe exactly the sequence
parts it holds."""
import ctypes
import random

import numpy as np
import pytest

from gdn_chunkwise_ut_gb300 import _lib


def _plan(bounds, C, parts):
    """[(n0, n1, offsets)] from the library's planner for sequences [a, b) given as bounds."""
    starts = np.array([bounds[0][0]] + [b for _, b in bounds], dtype=np.int64)
    nseq = len(bounds)
    cap_p, cap_cu = parts, nseq + 2 * parts
    out_b = np.zeros(2 * cap_p, dtype=np.int64)
    nsub = np.zeros(cap_p, dtype=np.int32)
    cu = np.zeros(cap_cu, dtype=np.int32)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    n = _lib.lib().kkt_test_plan_pieces(ptr(starts), nseq, C, parts, ptr(out_b), ptr(nsub), cap_p, ptr(cu), cap_cu)
    assert n >= 0
    plan, at = [], 0
    for p in range(n):
        offs = [int(x) for x in cu[at:at + nsub[p] + 1]]
        at += nsub[p] + 1
        plan.append((int(out_b[2 * p]), int(out_b[2 * p + 1]), offs))
    return plan


def _check(bounds, C, parts):
    plan = _plan(bounds, C, parts)
    total = sum(b - a for a, b in bounds)
    assert len(plan) <= parts
    assert sum(n1 - n0 for n0, n1, _ in plan) == total
    # consecutive, covering [first start, last end)
    assert plan[0][0] == bounds[0][0] and plan[-1][1] == bounds[-1][1]
    for (a0, a1, _), (b0, b1, _) in zip(plan, plan[1:]):
        assert a1 == b0
    for n0, n1, cu in plan:
        assert cu[0] == 0 and cu[-1] == n1 - n0 and all(x < y for x, y in zip(cu, cu[1:]))
        for x, y in zip(cu, cu[1:]):
            s0, s1 = n0 + x, n0 + y
            # the part [s0, s1) lies in one sequence and starts on a chunk boundary of it
            seq = next((a, b) for a, b in bounds if a <= s0 < b)
            assert s1 <= seq[1]
            assert (s0 - seq[0]) % C == 0
    return plan


@pytest.mark.parametrize("C", [32, 64, 128])
@pytest.mark.parametrize("parts", [1, 3, 8, 16])
def test_fixed_length_batch(C, parts):
    bounds = [(b * 8192, (b + 1) * 8192) for b in range(4)]
    plan = _check(bounds, C, parts)
    assert len(plan) == min(parts, 32768 // C)
    if parts == 8:
        assert all(n1 - n0 == 4096 for n0, n1, _ in plan)


@pytest.mark.parametrize("seed", range(5))
def test_varlen_batch(seed):
    rng = random.Random(seed)
    lengths = [rng.randint(0, 3000) for _ in range(rng.randint(1, 20))]
    lengths[0] = max(lengths[0], 1)
    bounds, pos = [], 0
    for n in lengths:
        bounds.append((pos, pos + n))
        pos += n
    for C in (32, 64, 128):
        for parts in (1, 2, 5, 8, 64):
            _check(bounds, C, parts)


def test_many_short_sequences_keep_the_limit():
    # sequences shorter than a chunk: pieces close early, the last one takes the rest
    bounds, pos = [], 0
    for n in [3, 70, 2, 130, 1, 65, 64, 5] * 6:
        bounds.append((pos, pos + n))
        pos += n
    for parts in (2, 3, 4):
        assert len(_check(bounds, 64, parts)) <= parts


def test_empty_batch():
    starts = np.zeros(2, dtype=np.int64)
    b, s, c = np.zeros(2, np.int64), np.zeros(1, np.int32), np.zeros(3, np.int32)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    assert _lib.lib().kkt_test_plan_pieces(ptr(starts), 1, 64, 1, ptr(b), ptr(s), 1, ptr(c), 3) == 0
